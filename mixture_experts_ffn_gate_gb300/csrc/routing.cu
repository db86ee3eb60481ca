// routing.cu -- router (top-k + softmax), the router projection for callers
// that pass the router weights, deterministic counting sort of the
// token->expert assignments and the fixed-order combine.
//
// Determinism: none of these kernels uses a floating-point atomic.  The sort
// uses integer shared-memory atomics only to count, and places every
// assignment at a position fixed by (expert, token, slot) -- the
// Mixture-of-Kittens article (section 결정론을 성능과 같은 급으로 올려놓은
// 선택) makes fixed accumulation order a design goal so that results do not
// depend on hardware scheduling.
#include "common.cuh"
#include "kernels.h"
#include "route_block.cuh"

namespace moe {

// ---------------------------------------------------------------- router
// One warp per token (route_token_warp): k rounds of a warp-wide maximum
// under a strict total order (larger logit first, smaller index on ties), so
// slot j holds the j-th pick; then the softmax over the k chosen logits.
constexpr int kRouterWarps = 8;

//
// On a workspace that keeps the fused decode kernel's state, block 0 also
// lowers that kernel's size word to tag_cap: this call's other regions
// (routing, act, the grouped path's act and z rows ...) start tag_cap words into the tag region,
// and a later fused call must not take what they leave there for tags.
__global__ void __launch_bounds__(32 * kRouterWarps) router_kernel(const float *__restrict__ logits, int T, int E,
                                                                   int k, int32_t *__restrict__ idx,
                                                                   float *__restrict__ w,
                                                                   int32_t *__restrict__ idx_copy,
                                                                   float *__restrict__ w_copy,
                                                                   unsigned long long *__restrict__ tag_size,
                                                                   unsigned long long tag_cap)
{
    extern __shared__ float vals[];  // [kRouterWarps][E]
    if (tag_size && blockIdx.x == 0 && threadIdx.x == 0 && *tag_size > tag_cap) *tag_size = tag_cap;
    const int t = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int e;
    float wt;
    route_token_warp(logits + (int64_t)t * E, E, k, vals + (threadIdx.x >> 5) * E, e, wt);
    const int j = threadIdx.x & 31;
    if (j < k) {
        idx[(int64_t)t * k + j] = e;
        w[(int64_t)t * k + j] = wt;
        if (idx_copy) idx_copy[(int64_t)t * k + j] = e;
        if (w_copy) w_copy[(int64_t)t * k + j] = wt;
    }
}

// ---------------------------------------------------------------- router projection
// logits[t, e] = round_f32(sum_h x[t, h] * W_r[e, h] + b[e]), one warp per
// logit (router_logit_warp), for calls that pass the router weights instead
// of logits and do not take the fused decode kernel.
__global__ void __launch_bounds__(32 * kRouterWarps) router_gemv_kernel(const uint16_t *__restrict__ x,
                                                                        const uint16_t *__restrict__ wr,
                                                                        const float *__restrict__ bias, int T,
                                                                        int H, int E, float *__restrict__ logits,
                                                                        float *__restrict__ logits_copy)
{
    const int64_t o = (int64_t)blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
    if (o >= (int64_t)T * E) return;
    const int t = (int)(o / E), e = (int)(o - (int64_t)t * E);
    const float v = router_logit_warp(x + (int64_t)t * H, wr + (int64_t)e * H, H, bias ? __ldg(bias + e) : 0.0f,
                                      threadIdx.x & 31);
    if ((threadIdx.x & 31) == 0) {
        logits[o] = v;
        if (logits_copy) logits_copy[o] = v;
    }
}

// ---------------------------------------------------------------- sort
// Single block of SORT_THREADS threads.  Warp q owns a contiguous range of
// assignments (a = t*k + j).  Pass 1 counts per (warp, expert); a scan turns
// the counts into expert-major offsets and per-warp bases; pass 2 walks each
// range in order and places assignment a at
//   offs[e] + (assignments of e in earlier warps) + (earlier ones in this warp),
// i.e. the assignments of each expert end up in ascending a = token order.
// With pad > 1 every expert's segment is rounded up to a multiple of pad
// rows (offs are the padded offsets, the pad rows' perm is -1) and counts[e]
// (nullable) gets the expert's number of assignments.
constexpr int SORT_THREADS = 1024;
constexpr int SORT_WARPS = SORT_THREADS / 32;

__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch /*[SORT_WARPS+1]*/, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = lane < SORT_WARPS ? scratch[lane] : 0;
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += n;
        }
        if (lane < SORT_WARPS) scratch[lane] = si - s;
        if (lane == SORT_WARPS - 1) scratch[SORT_WARPS] = si;
    }
    __syncthreads();
    const int r = scratch[warp] + incl - v;
    *total = scratch[SORT_WARPS];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(SORT_THREADS) sort_kernel(const int32_t *__restrict__ idx, int n_assign, int E,
                                                           int chunk_max, int32_t *__restrict__ offs,
                                                           int32_t *__restrict__ perm, int32_t *__restrict__ pos,
                                                           int32_t *__restrict__ uexp, int32_t *__restrict__ ucount,
                                                           int4 *__restrict__ chunks, int32_t *__restrict__ nchunks,
                                                           int pad, int32_t *__restrict__ counts)
{
    extern __shared__ int hist[];  // [SORT_WARPS][E]
    __shared__ int scratch[SORT_WARPS + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < SORT_WARPS * E; i += SORT_THREADS) hist[i] = 0;
    __syncthreads();
    const int per = (n_assign + SORT_WARPS - 1) / SORT_WARPS;
    const int a_begin = min(n_assign, warp * per), a_end = min(n_assign, a_begin + per);
    for (int a = a_begin + lane; a < a_end; a += 32) atomicAdd(&hist[warp * E + idx[a]], 1);
    __syncthreads();

    // E <= SORT_THREADS: thread e owns expert e
    const int e = tid;
    int cnt = 0;
    if (e < E)
        for (int q = 0; q < SORT_WARPS; ++q) cnt += hist[q * E + e];
    int total;
    const int padded = (cnt + pad - 1) / pad * pad;
    const int off = block_exclusive_scan(e < E ? padded : 0, scratch, &total);
    if (e < E) {
        offs[e] = off;
        if (e == E - 1) offs[E] = off + padded;
        if (counts) counts[e] = cnt;
        for (int p = off + cnt; p < off + padded; ++p) perm[p] = -1;
        int run = off;
        for (int q = 0; q < SORT_WARPS; ++q) {
            const int h = hist[q * E + e];
            hist[q * E + e] = run;
            run += h;
        }
    }
    // touched experts, ascending
    const int touched = (e < E && cnt > 0) ? 1 : 0;
    int n_touched;
    const int slot = block_exclusive_scan(touched, scratch, &n_touched);
    if (touched) uexp[slot] = e;
    if (tid == 0) *ucount = n_touched;
    // row chunks of at most chunk_max assignments per expert (grouped GEMMs):
    // {expert, first sorted row, rows, index of the expert's first chunk}
    if (chunks) {
        const int nch = (e < E) ? (cnt + chunk_max - 1) / chunk_max : 0;
        int n_total;
        const int c0 = block_exclusive_scan(nch, scratch, &n_total);
        for (int c = 0; c < nch; ++c)
            chunks[c0 + c] = make_int4(e, off + c * chunk_max, min(chunk_max, cnt - c * chunk_max), c0);
        if (tid == 0) *nchunks = n_total;
    }
    __syncthreads();

    // pass 2: stable placement
    const unsigned lt = (1u << lane) - 1u;
    for (int base = a_begin; base < a_end; base += 32) {
        const int a = base + lane;
        const bool valid = a < a_end;
        const int ea = valid ? idx[a] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, ea);
        const int rank = __popc(same & lt);
        int p = 0;
        if (valid) {
            p = hist[warp * E + ea] + rank;
            perm[p] = a;
            pos[a] = p;
        }
        __syncwarp();
        if (valid && rank == 0) hist[warp * E + ea] += __popc(same);
        __syncwarp();
    }
}

// ---------------------------------------------------------------- combine
// out[t, h] = sum_{j ascending} w[t,j] * z[pos[t*k+j], h]   (FP32, fixed order);
// with w null the rows are summed unweighted (the backward pass's dx)
constexpr int kCombineBatch = 8;   // slots whose rows one thread loads together

__global__ void combine_kernel(const float *__restrict__ z, const float *__restrict__ w,
                               const int32_t *__restrict__ pos, int T, int H, int k, float *__restrict__ out)
{
    const int hv = H / 4;
    const int64_t total = (int64_t)T * hv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / hv), c = (int)(i - (int64_t)t * hv);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        auto add = [&](float wj, const float4 &v) {
            acc.x = fmaf(wj, v.x, acc.x);
            acc.y = fmaf(wj, v.y, acc.y);
            acc.z = fmaf(wj, v.z, acc.z);
            acc.w = fmaf(wj, v.w, acc.w);
        };
        if (k <= kCombineBatch) {
            // every slot's row load in flight at once; the sum keeps slot order
            float4 v[kCombineBatch];
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j)
                if (j < k) v[j] = ld_nc_f4(z + (int64_t)__ldg(pos + (int64_t)t * k + j) * H + 4 * c);
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j)
                if (j < k) add(w ? __ldg(w + (int64_t)t * k + j) : 1.0f, v[j]);
        } else {
            for (int j = 0; j < k; ++j)
                add(w ? __ldg(w + (int64_t)t * k + j) : 1.0f,
                    ld_nc_f4(z + (int64_t)__ldg(pos + (int64_t)t * k + j) * H + 4 * c));
        }
        reinterpret_cast<float4 *>(out)[i] = acc;
    }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_router(const float *logits, int T, int E, int k, int32_t *idx, float *w, int32_t *idx_copy,
                          float *w_copy, unsigned long long *tag_size, unsigned long long tag_cap, cudaStream_t s)
{
    router_kernel<<<(unsigned)ceil_div(T, kRouterWarps), 32 * kRouterWarps, (size_t)kRouterWarps * E * 4, s>>>(
        logits, T, E, k, idx, w, idx_copy, w_copy, tag_size, tag_cap);
    return cudaPeekAtLastError();
}

cudaError_t launch_router_gemv(const void *x, const void *wr, const float *bias, int T, int H, int E, float *logits,
                               float *logits_copy, cudaStream_t s)
{
    const int64_t n = (int64_t)T * E;
    router_gemv_kernel<<<(unsigned)ceil_div(n, kRouterWarps), 32 * kRouterWarps, 0, s>>>(
        (const uint16_t *)x, (const uint16_t *)wr, bias, T, H, E, logits, logits_copy);
    return cudaPeekAtLastError();
}

size_t sort_smem_bytes(int E) { return (size_t)SORT_WARPS * E * sizeof(int); }

cudaError_t routing_init_device()
{
    return cudaFuncSetAttribute(sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sort_smem_bytes(1024));
}

cudaError_t launch_sort(const int32_t *idx, int n_assign, int E, int chunk_max, int32_t *offs, int32_t *perm,
                        int32_t *pos, int32_t *uexp, int32_t *ucount, int4 *chunks, int32_t *nchunks,
                        cudaStream_t s, int pad, int32_t *counts)
{
    const size_t smem = sort_smem_bytes(E);
    sort_kernel<<<1, SORT_THREADS, smem, s>>>(idx, n_assign, E, chunk_max, offs, perm, pos, uexp, ucount, chunks,
                                              nchunks, pad, counts);
    return cudaPeekAtLastError();
}

cudaError_t launch_combine(const float *z, const float *w, const int32_t *pos, int T, int H, int k, float *out,
                           int n_sm, cudaStream_t s)
{
    const int64_t total = (int64_t)T * (H / 4);
    const int64_t blocks = ceil_div(total, 256);
    const int grid = (int)(blocks < (int64_t)n_sm * 8 ? blocks : (int64_t)n_sm * 8);
    combine_kernel<<<grid, 256, 0, s>>>(z, w, pos, T, H, k, out);
    return cudaPeekAtLastError();
}

}  // namespace moe
