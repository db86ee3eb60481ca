// decode1.cu -- the decode path for a single token (T = 1), as two kernels.
//
// The warp-decode article ("Cursor warp decode 공개 ...", section 핵심 내용)
// finishes a decode step in two kernels, one warp per output scalar, summing
// the routed experts' contributions in FP32 with no padding, scatter or
// per-expert buffers; its section 경쟁 구도 / 비교 keeps the intermediate
// activation unquantised.  On GB300 the two kernels here are persistent, one
// CTA of each per SM, and move the weights with bulk copies:
//   decode1_gate_up: every CTA routes the token itself (the router kernel's
//     rank-based top-k and softmax, same bits) and owns an equal, contiguous
//     share of the k*2I gate/up rows of the chosen experts.  Within one expert
//     those rows are contiguous in memory, so a producer warp moves them into
//     a shared-memory ring as bulk copies (cp.async.bulk) of whole rows,
//     about 16 KB each; consumer warps take the rows round-robin and write
//     each row's dot product with x (FP32) to gu[slot][row].
//   decode1_down: launched as a programmatic dependent of gate_up, which lets
//     it go as soon as gate_up has routed.  The two kernels are sized to share
//     an SM, so the down CTA's producer streams W_down[e_j, h_lo:h_hi, :]
//     (contiguous per expert; the weights do not depend on gate_up) while
//     gate_up is still streaming.  Its consumers wait for gate_up, form
//     act = silu(gate) * up in shared memory (FP32), dot each row with act[j]
//     and finally sum out[h] = sum_j w_j * part[h][j] in slot order.
// Each dot product uses decode.cu's lane split, chunk order, fmaf order and
// shuffle butterfly, so this path returns the same bits as the general decode
// path.  Every consumer warp visits every chunk in order, so a ring slot's
// parity waits are never more than one phase ahead; every wait is bounded.
#include <atomic>
#include <random>

#include "common.cuh"
#include "kernels.h"
#include "route_block.cuh"
#include "sm100_ptx.cuh"

namespace moe {

__device__ uint32_t g_decode1_fault_word = 0;

namespace {

// Registers: 2 CTAs x 416 threads x <= 78 fit one SM's 64 K.
constexpr int kConsumers = 12;
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kSlotTarget = 16 * 1024;  // bytes per bulk copy (whole rows)
constexpr int kMaxSlots = 16;
constexpr int kSmemCap = 226 * 1024;    // dynamic, one CTA; the per-block limit also covers static smem
constexpr int kSmemPerSm = 224 * 1024;  // dynamic, both CTAs together
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;

__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

// Shared-memory layout: ring | full[slots] | empty[slots] | flag | keys[E] | payload
struct Layout {
    uint32_t full, empty, flag, keys, payload, total;
};

__host__ __device__ inline Layout layout(int slots, int slot_bytes, int E, uint32_t payload_bytes)
{
    Layout L;
    uint32_t o = (uint32_t)slots * slot_bytes;
    L.full = o;
    o += slots * 8;
    L.empty = o;
    o += slots * 8;
    L.flag = o;
    o += 16;
    L.keys = o;
    o = align16(o + (uint32_t)E * 8);
    L.payload = o;
    L.total = o + payload_bytes;
    return L;
}

__device__ __forceinline__ void fail(volatile int *flag, uint32_t bit)
{
    if (!*flag) atomicOr(&g_decode1_fault_word, bit);
    *flag = 1;
}

__device__ __forceinline__ uint4 lds16(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

__device__ __forceinline__ void init_ring(uint64_t *full, uint64_t *empty, int slots, volatile int *flag)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < slots; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, kConsumers);
        }
        *flag = 0;
        ptx::fence_barrier_init();
    }
}

// The producer waits (bounded) until the last `slots` chunks it issued have
// landed, so no copy is in flight when the CTA exits.
__device__ __forceinline__ void drain(uint64_t *full, int slots, int issued)
{
    const volatile int keep = 0;
    for (int c = issued - 1; c >= 0 && c >= issued - slots; --c)
        ptx::mbar_wait_bounded(full + (c % slots), (uint32_t)(c / slots) & 1, &keep, kDrainNs);
}

// First row t >= t0 of the CTA's row sequence (starting at lo) that belongs
// to consumer warp cw (rows go round-robin over the consumer warps).
__device__ __forceinline__ int first_row(int t0, int lo, int cw)
{
    const int m = (t0 - lo) % kConsumers;
    return t0 + ((cw - m) % kConsumers + kConsumers) % kConsumers;
}

// ------------------------------------------------------------------ gate_up
// Rows r in [0, k*2I): slot j = r / 2I, row q = r % 2I of expert sel[j]'s
// [2I, H] block.  A chunk is at most rpc rows and never crosses an expert.
__device__ __forceinline__ int gu_chunk_end(int t0, int hi, int per_expert, int rpc)
{
    const int e_end = (t0 / per_expert + 1) * per_expert;
    return min(hi, min(e_end, t0 + rpc));
}

__global__ void __launch_bounds__(kThreads, 2)
    decode1_gate_up_kernel(const uint16_t *__restrict__ x, const float *__restrict__ logits,
                           const uint16_t *__restrict__ wgu, int H, int I, int E, int k, int slots, int rpc,
                           float *__restrict__ gu, int32_t *__restrict__ idx_out, float *__restrict__ w_out)
{
    extern __shared__ __align__(128) uint8_t sm[];
    const int slot_bytes = rpc * 2 * H;
    const Layout L = layout(slots, slot_bytes, E, (uint32_t)H * 4);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(sm + L.empty);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + L.flag);
    // x in FP32, two planes: element 8u+e sits in plane e/4 at 4u + e%4, so a
    // lane's 8 consecutive elements are two float4 loads that are contiguous
    // across the warp (no bank conflicts, no per-row unpacking)
    float *xs = reinterpret_cast<float *>(sm + L.payload);
    __shared__ int sel[32];
    __shared__ float wsm[32];

    init_ring(full, empty, slots, flag);
    route_token_block(logits, E, k, reinterpret_cast<unsigned long long *>(sm + L.keys), sel, wsm);
    if (blockIdx.x == 0 && threadIdx.x < k) {
        if (idx_out) idx_out[threadIdx.x] = sel[threadIdx.x];
        if (w_out) w_out[threadIdx.x] = wsm[threadIdx.x];
    }
    pdl_trigger();

    const int per_expert = 2 * I;
    const int rows = k * per_expert;
    const int lo = (int)((int64_t)rows * blockIdx.x / gridDim.x);
    const int hi = (int)((int64_t)rows * (blockIdx.x + 1) / gridDim.x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        if (lane == 0) {
            int c = 0;
            for (int t0 = lo; t0 < hi; ++c) {
                const int t1 = gu_chunk_end(t0, hi, per_expert, rpc);
                const int s = c % slots;
                if (!ptx::mbar_wait_bounded(empty + s, ((uint32_t)(c / slots) & 1) ^ 1, flag, kWaitNs)) {
                    fail(flag, 1u);
                    break;
                }
                const int j = t0 / per_expert, q0 = t0 - j * per_expert;
                const uint32_t bytes = (uint32_t)(t1 - t0) * 2 * H;
                ptx::mbar_arrive_expect_tx(full + s, bytes);
                ptx::bulk_load(sm + (size_t)s * slot_bytes, wgu + ((int64_t)sel[j] * per_expert + q0) * H, bytes,
                               full + s);
                t0 = t1;
            }
            drain(full, slots, c);
        }
        return;
    }

    // consumers stage x while the first copies are in flight
    for (int u = threadIdx.x - 32; u < H / 8; u += kConsumers * 32) {
        float f[8];
        unpack8(ld_nc16(x + (size_t)u * 8), f);
        *reinterpret_cast<float4 *>(xs + 4 * u) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4 *>(xs + H / 2 + 4 * u) = make_float4(f[4], f[5], f[6], f[7]);
    }
    ptx::named_sync(1, kConsumers * 32);

    const int cw = warp - 1;
    int c = 0;
    for (int t0 = lo; t0 < hi; ++c) {
        const int t1 = gu_chunk_end(t0, hi, per_expert, rpc);
        const int s = c % slots;
        if (!ptx::mbar_wait_bounded(full + s, (uint32_t)(c / slots) & 1, flag, kWaitNs)) {
            fail(flag, 2u);
            break;
        }
        const uint8_t *chunk = sm + (size_t)s * slot_bytes;
        for (int t = first_row(t0, lo, cw); t < t1; t += kConsumers) {
            const uint8_t *row = chunk + (size_t)(t - t0) * 2 * H;
            float acc = 0.0f;
#pragma unroll 4
            for (int h = lane * 8; h < H; h += 256) {
                float wf[8], xf[8];
                unpack8(lds16(row + 2 * h), wf);
                const float4 x0 = *reinterpret_cast<const float4 *>(xs + h / 2);
                const float4 x1 = *reinterpret_cast<const float4 *>(xs + H / 2 + h / 2);
                xf[0] = x0.x; xf[1] = x0.y; xf[2] = x0.z; xf[3] = x0.w;
                xf[4] = x1.x; xf[5] = x1.y; xf[6] = x1.z; xf[7] = x1.w;
#pragma unroll
                for (int q = 0; q < 8; ++q) acc = fmaf(wf[q], xf[q], acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) gu[t] = acc;  // t = j * 2I + q
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + s);
        t0 = t1;
    }
}

// ------------------------------------------------------------------ down
// CTA rows: for slot j = 0..k-1, dims h in [h_lo, h_hi) in chunks of at most
// rpd rows (contiguous in W_down[e_j]).  Row sequence index = j * nh + (h - h_lo).
__global__ void __launch_bounds__(kThreads, 2)
    decode1_down_kernel(const float *__restrict__ gu, const float *__restrict__ logits,
                        const uint16_t *__restrict__ wd, int H, int I, int E, int k, int slots, int rpd, int nh_max,
                        float *__restrict__ out)
{
    extern __shared__ __align__(128) uint8_t sm[];
    const int slot_bytes = rpd * 2 * I;
    const Layout L = layout(slots, slot_bytes, E, (uint32_t)(k * I + nh_max * k) * 4);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(sm + L.empty);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + L.flag);
    float *act = reinterpret_cast<float *>(sm + L.payload);  // [k][I]
    float *part = act + (size_t)k * I;                        // [nh][k]
    __shared__ int sel[32];
    __shared__ float wsm[32];

    init_ring(full, empty, slots, flag);
    route_token_block(logits, E, k, reinterpret_cast<unsigned long long *>(sm + L.keys), sel, wsm);

    const int h_lo = (int)((int64_t)H * blockIdx.x / gridDim.x);
    const int h_hi = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
    const int nh = h_hi - h_lo;
    const int cpe = (nh + rpd - 1) / rpd;  // chunks per expert
    const int n_chunks = k * cpe;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        // the weights do not depend on gate_up: stream them now
        if (lane == 0) {
            int c = 0;
            for (; c < n_chunks; ++c) {
                const int j = c / cpe, h0 = h_lo + (c - j * cpe) * rpd;
                const int nr = min(rpd, h_hi - h0);
                const int s = c % slots;
                if (!ptx::mbar_wait_bounded(empty + s, ((uint32_t)(c / slots) & 1) ^ 1, flag, kWaitNs)) {
                    fail(flag, 4u);
                    break;
                }
                const uint32_t bytes = (uint32_t)nr * 2 * I;
                ptx::mbar_arrive_expect_tx(full + s, bytes);
                ptx::bulk_load(sm + (size_t)s * slot_bytes, wd + ((int64_t)sel[j] * H + h0) * I, bytes, full + s);
            }
            drain(full, slots, c);
        }
        return;
    }

    // consumers: act = silu(gate) * up for the k slots, from gate_up's output
    pdl_wait();
    const int ct = threadIdx.x - 32, n_ct = kConsumers * 32;
    const int n4 = k * I / 4;
    for (int v0 = ct; v0 < n4; v0 += 4 * n_ct) {
        float4 g4[4], u4[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int v = v0 + b * n_ct;
            if (v < n4) {
                const int j = (4 * v) / I, i = 4 * v - j * I;
                g4[b] = *reinterpret_cast<const float4 *>(gu + (size_t)j * 2 * I + i);
                u4[b] = *reinterpret_cast<const float4 *>(gu + (size_t)j * 2 * I + I + i);
            }
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int v = v0 + b * n_ct;
            if (v < n4) {
                float4 a;
                a.x = swiglu(g4[b].x, u4[b].x);
                a.y = swiglu(g4[b].y, u4[b].y);
                a.z = swiglu(g4[b].z, u4[b].z);
                a.w = swiglu(g4[b].w, u4[b].w);
                // row j in two planes (element 8u+e at plane e/4, offset 4u + e%4)
                const int j = (4 * v) / I, i = 4 * v - j * I;
                *reinterpret_cast<float4 *>(act + (size_t)j * I + ((i >> 2) & 1) * (I / 2) + (i >> 3) * 4) = a;
            }
        }
    }
    ptx::named_sync(1, n_ct);

    const int cw = warp - 1;
    for (int c = 0; c < n_chunks; ++c) {
        const int j = c / cpe, h0 = h_lo + (c - j * cpe) * rpd;
        const int nr = min(rpd, h_hi - h0);
        const int s = c % slots;
        if (!ptx::mbar_wait_bounded(full + s, (uint32_t)(c / slots) & 1, flag, kWaitNs)) {
            fail(flag, 8u);
            break;
        }
        const uint8_t *chunk = sm + (size_t)s * slot_bytes;
        const float *arow = act + (size_t)j * I;
        const int base = j * nh + (h0 - h_lo);  // row sequence index of the chunk's first row
        for (int u = first_row(base, 0, cw) - base; u < nr; u += kConsumers) {
            const uint8_t *row = chunk + (size_t)u * 2 * I;
            float acc = 0.0f;
#pragma unroll 4
            for (int i = lane * 8; i < I; i += 256) {
                float wf[8];
                unpack8(lds16(row + 2 * i), wf);
                const float4 v0 = *reinterpret_cast<const float4 *>(arow + i / 2);
                const float4 v1 = *reinterpret_cast<const float4 *>(arow + I / 2 + i / 2);
                const float af[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int q = 0; q < 8; ++q) acc = fmaf(wf[q], af[q], acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) part[(h0 - h_lo + u) * k + j] = acc;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + s);
    }
    ptx::named_sync(1, n_ct);
    if (*flag) return;
    for (int q = ct; q < nh; q += n_ct) {
        float o = 0.0f;
        for (int j = 0; j < k; ++j) o = fmaf(wsm[j], part[q * k + j], o);
        out[h_lo + q] = o;
    }
}

// ------------------------------------------------------------------ fused
// The single-token layer in one cooperative launch (all CTAs resident, one
// per SM).  Each CTA routes the token once; its producer streams first the
// CTA's share of gate/up rows, then -- without a pause, since W_down does not
// depend on gate_up -- its W_down rows, through one ring.  The consumers
// compute the gate/up dot products (gu), meet the other CTAs at a grid-wide
// barrier, form act = silu(gate) * up in shared memory (reusing the space of
// x), and finish the down rows, many of which are already in the ring.
//
// Grid barrier: CTA b stores the call's epoch (a 64-bit value unique to the
// call) into flags[b] with release semantics once its gu rows are written,
// then waits (bounded) until every flags[c] holds the epoch.  Stale values
// from earlier calls never equal a later epoch, so nothing needs zeroing.
constexpr int kFusedConsumers = 16;
constexpr int kFusedThreads = 32 * (1 + kFusedConsumers);

__device__ __forceinline__ int fused_first_row(int t0, int lo, int cw)
{
    const int m = (t0 - lo) % kFusedConsumers;
    return t0 + ((cw - m) % kFusedConsumers + kFusedConsumers) % kFusedConsumers;
}

__global__ void __launch_bounds__(kFusedThreads, 1)
    decode1_fused_kernel(const uint16_t *__restrict__ x, const float *__restrict__ logits,
                         const uint16_t *__restrict__ wgu, const uint16_t *__restrict__ wd, int H, int I, int E,
                         int k, int slots, int slot_bytes, int rpc, int rpd, int nh_max, float *__restrict__ gu,
                         unsigned long long *__restrict__ flags, unsigned long long epoch,
                         int32_t *__restrict__ idx_out, float *__restrict__ w_out, float *__restrict__ out)
{
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t xa_bytes = (uint32_t)(4 * H > 4 * k * I ? 4 * H : 4 * k * I);  // x, later act
    const Layout L = layout(slots, slot_bytes, E, xa_bytes + (uint32_t)nh_max * k * 4);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(sm + L.empty);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + L.flag);
    float *xs = reinterpret_cast<float *>(sm + L.payload);   // phase A: x, two planes
    float *act = xs;                                          // phase B: act [k][I], two planes per row
    float *part = reinterpret_cast<float *>(sm + L.payload + xa_bytes);  // [nh][k]
    __shared__ int sel[32];
    __shared__ float wsm[32];
    if (threadIdx.x == 0) {
        for (int s = 0; s < slots; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, kFusedConsumers);
        }
        *flag = 0;
        ptx::fence_barrier_init();
    }
    route_token_block(logits, E, k, reinterpret_cast<unsigned long long *>(sm + L.keys), sel, wsm);
    if (blockIdx.x == 0 && threadIdx.x < k) {
        if (idx_out) idx_out[threadIdx.x] = sel[threadIdx.x];
        if (w_out) w_out[threadIdx.x] = wsm[threadIdx.x];
    }

    // phase A rows: [lo, hi) of the k*2I gate/up rows; phase B: output dims
    // [h_lo, h_hi), all k slots, cpe chunks of <= rpd rows per slot
    const int per_expert = 2 * I;
    const int rows = k * per_expert;
    const int lo = (int)((int64_t)rows * blockIdx.x / gridDim.x);
    const int hi = (int)((int64_t)rows * (blockIdx.x + 1) / gridDim.x);
    const int h_lo = (int)((int64_t)H * blockIdx.x / gridDim.x);
    const int h_hi = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
    const int nh = h_hi - h_lo;
    const int cpe = (nh + rpd - 1) / rpd;
    const int nb = k * cpe;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        if (lane == 0) {
            int c = 0;
            bool ok = true;
            for (int t0 = lo; t0 < hi && ok; ++c) {
                const int t1 = gu_chunk_end(t0, hi, per_expert, rpc);
                const int s = c % slots;
                if (!ptx::mbar_wait_bounded(empty + s, ((uint32_t)(c / slots) & 1) ^ 1, flag, kWaitNs)) {
                    fail(flag, 16u);
                    ok = false;
                    break;
                }
                const int j = t0 / per_expert, q0 = t0 - j * per_expert;
                const uint32_t bytes = (uint32_t)(t1 - t0) * 2 * H;
                ptx::mbar_arrive_expect_tx(full + s, bytes);
                ptx::bulk_load(sm + (size_t)s * slot_bytes, wgu + ((int64_t)sel[j] * per_expert + q0) * H, bytes,
                               full + s);
                t0 = t1;
            }
            for (int q = 0; q < nb && ok; ++q, ++c) {
                const int j = q / cpe, h0 = h_lo + (q - j * cpe) * rpd;
                const int nr = min(rpd, h_hi - h0);
                const int s = c % slots;
                if (!ptx::mbar_wait_bounded(empty + s, ((uint32_t)(c / slots) & 1) ^ 1, flag, kWaitNs)) {
                    fail(flag, 16u);
                    ok = false;
                    break;
                }
                const uint32_t bytes = (uint32_t)nr * 2 * I;
                ptx::mbar_arrive_expect_tx(full + s, bytes);
                ptx::bulk_load(sm + (size_t)s * slot_bytes, wd + ((int64_t)sel[j] * H + h0) * I, bytes, full + s);
            }
            drain(full, slots, c);
        }
        return;
    }

    const int ct = threadIdx.x - 32, n_ct = kFusedConsumers * 32;
    const int cw = warp - 1;
    for (int u = ct; u < H / 8; u += n_ct) {
        float f[8];
        unpack8(ld_nc16(x + (size_t)u * 8), f);
        *reinterpret_cast<float4 *>(xs + 4 * u) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4 *>(xs + H / 2 + 4 * u) = make_float4(f[4], f[5], f[6], f[7]);
    }
    ptx::named_sync(1, n_ct);

    // phase A: gate/up row dot products
    int c = 0;
    for (int t0 = lo; t0 < hi; ++c) {
        const int t1 = gu_chunk_end(t0, hi, per_expert, rpc);
        const int s = c % slots;
        if (!ptx::mbar_wait_bounded(full + s, (uint32_t)(c / slots) & 1, flag, kWaitNs)) {
            fail(flag, 32u);
            break;
        }
        const uint8_t *chunk = sm + (size_t)s * slot_bytes;
        for (int t = fused_first_row(t0, lo, cw); t < t1; t += kFusedConsumers) {
            const uint8_t *row = chunk + (size_t)(t - t0) * 2 * H;
            float acc = 0.0f;
#pragma unroll 4
            for (int h = lane * 8; h < H; h += 256) {
                float wf[8];
                unpack8(lds16(row + 2 * h), wf);
                const float4 x0 = *reinterpret_cast<const float4 *>(xs + h / 2);
                const float4 x1 = *reinterpret_cast<const float4 *>(xs + H / 2 + h / 2);
                const float xf[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int q = 0; q < 8; ++q) acc = fmaf(wf[q], xf[q], acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) gu[t] = acc;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + s);
        t0 = t1;
    }

    // grid barrier: every CTA's gu rows written and visible
    __threadfence();
    ptx::named_sync(1, n_ct);
    if (ct == 0 && !*flag) ptx::st_release_gpu(flags + blockIdx.x, epoch);
    // consumer thread ct watches the flags of CTAs ct, ct + n_ct, ... (all in parallel)
    const uint64_t t_start = ptx::globaltimer_ns();
    for (int b = ct; b < (int)gridDim.x && !*flag; b += n_ct) {
        for (uint32_t spin = 0; ptx::ld_acquire_gpu(flags + b) != epoch; ++spin) {
            if ((spin & 63) == 63 && (*flag || ptx::globaltimer_ns() - t_start > kWaitNs)) {
                if (!*flag) fail(flag, 64u);
                break;
            }
        }
    }
    ptx::named_sync(1, n_ct);
    __threadfence();
    if (*flag) return;

    // act = silu(gate) * up for the k slots, two planes per row (x's space)
    const int n4 = k * I / 4;
    for (int v0 = ct; v0 < n4; v0 += 4 * n_ct) {
        float4 g4[4], u4[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int v = v0 + b * n_ct;
            if (v < n4) {
                const int j = (4 * v) / I, i = 4 * v - j * I;
                g4[b] = __ldcg(reinterpret_cast<const float4 *>(gu + (size_t)j * 2 * I + i));
                u4[b] = __ldcg(reinterpret_cast<const float4 *>(gu + (size_t)j * 2 * I + I + i));
            }
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int v = v0 + b * n_ct;
            if (v < n4) {
                const int j = (4 * v) / I, i = 4 * v - j * I;
                float4 a;
                a.x = swiglu(g4[b].x, u4[b].x);
                a.y = swiglu(g4[b].y, u4[b].y);
                a.z = swiglu(g4[b].z, u4[b].z);
                a.w = swiglu(g4[b].w, u4[b].w);
                *reinterpret_cast<float4 *>(act + (size_t)j * I + ((i >> 2) & 1) * (I / 2) + (i >> 3) * 4) = a;
            }
        }
    }
    ptx::named_sync(1, n_ct);

    // phase B: W_down rows
    for (int q = 0; q < nb; ++q, ++c) {
        const int j = q / cpe, h0 = h_lo + (q - j * cpe) * rpd;
        const int nr = min(rpd, h_hi - h0);
        const int s = c % slots;
        if (!ptx::mbar_wait_bounded(full + s, (uint32_t)(c / slots) & 1, flag, kWaitNs)) {
            fail(flag, 128u);
            break;
        }
        const uint8_t *chunk = sm + (size_t)s * slot_bytes;
        const float *arow = act + (size_t)j * I;
        const int base = j * nh + (h0 - h_lo);
        for (int u = fused_first_row(base, 0, cw) - base; u < nr; u += kFusedConsumers) {
            const uint8_t *row = chunk + (size_t)u * 2 * I;
            float acc = 0.0f;
#pragma unroll 4
            for (int i = lane * 8; i < I; i += 256) {
                float wf[8];
                unpack8(lds16(row + 2 * i), wf);
                const float4 v0 = *reinterpret_cast<const float4 *>(arow + i / 2);
                const float4 v1 = *reinterpret_cast<const float4 *>(arow + I / 2 + i / 2);
                const float af[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) acc = fmaf(wf[qq], af[qq], acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) part[(h0 - h_lo + u) * k + j] = acc;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + s);
    }
    ptx::named_sync(1, n_ct);
    if (*flag) return;
    for (int qh = ct; qh < nh; qh += n_ct) {
        float o = 0.0f;
        for (int j = 0; j < k; ++j) o = fmaf(wsm[j], part[qh * k + j], o);
        out[h_lo + qh] = o;
    }
}

// Ring geometry of both kernels: whole rows per slot (about kSlotTarget
// bytes), and as many slots as fit -- preferably with both kernels' CTAs on
// one SM together, otherwise each alone.
struct Plan {
    int rpc, rpd, slots_a, slots_b, nh_max;
    uint32_t payload_a, payload_b;
    bool together;
};

Plan plan_for(int H, int I, int E, int k, int n_sm)
{
    Plan p;
    p.nh_max = (H + n_sm - 1) / n_sm;
    p.rpc = kSlotTarget / (2 * H) > 0 ? kSlotTarget / (2 * H) : 1;
    p.rpd = kSlotTarget / (2 * I) > 0 ? kSlotTarget / (2 * I) : 1;
    if (p.rpd > p.nh_max) p.rpd = p.nh_max > 0 ? p.nh_max : 1;
    const int sa = p.rpc * 2 * H, sb = p.rpd * 2 * I;
    p.payload_a = (uint32_t)H * 4;
    p.payload_b = (uint32_t)(k * I + p.nh_max * k) * 4;
    const int fa = (int)layout(0, sa, E, p.payload_a).total + 2 * kMaxSlots * 8;
    const int fb = (int)layout(0, sb, E, p.payload_b).total + 2 * kMaxSlots * 8;
    const auto cap = [](int n) { return n > kMaxSlots ? kMaxSlots : n; };
    // together: split the ring bytes in proportion to the weight bytes (2:1)
    const int ring = kSmemPerSm - fa - fb;
    p.slots_a = cap(ring * 2 / 3 / sa);
    p.slots_b = cap((ring - p.slots_a * sa) / sb);
    p.together = p.slots_a >= 2 && p.slots_b >= 2;
    if (!p.together) {
        p.slots_a = cap((kSmemCap - fa) / sa);
        p.slots_b = cap((kSmemCap - fb) / sb);
    }
    return p;
}

// Fused kernel geometry: one ring for both phases, slots sized for the larger
// of a gate/up chunk and a down chunk.
struct FusedPlan {
    int rpc, rpd, slot_bytes, slots, nh_max;
    uint32_t payload;
};

FusedPlan fused_plan_for(int H, int I, int E, int k, int n_sm)
{
    FusedPlan p;
    p.nh_max = (H + n_sm - 1) / n_sm;
    p.rpc = kSlotTarget / (2 * H) > 0 ? kSlotTarget / (2 * H) : 1;
    p.rpd = kSlotTarget / (2 * I) > 0 ? kSlotTarget / (2 * I) : 1;
    if (p.rpd > p.nh_max) p.rpd = p.nh_max > 0 ? p.nh_max : 1;
    p.slot_bytes = p.rpc * 2 * H > p.rpd * 2 * I ? p.rpc * 2 * H : p.rpd * 2 * I;
    const int xa = 4 * H > 4 * k * I ? 4 * H : 4 * k * I;
    p.payload = (uint32_t)(xa + p.nh_max * k * 4);
    const int fixed = (int)layout(0, p.slot_bytes, E, p.payload).total + 2 * kMaxSlots * 8;
    const int n = (kSmemCap - fixed) / p.slot_bytes;
    p.slots = n > kMaxSlots ? kMaxSlots : n;
    return p;
}

std::atomic<unsigned long long> g_epoch{0};

// A value unique to this call: a 64-bit counter whose start is drawn at random
// once per process, so flags left in a workspace by earlier calls (or by
// another process) do not match it.
unsigned long long next_epoch()
{
    static const unsigned long long base = [] {
        std::random_device rd;
        return ((unsigned long long)rd() << 32) ^ rd() ^ 0x9e3779b97f4a7c15ull;
    }();
    return base + 2 * g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
}

}  // namespace

bool decode1_fused_supported(int H, int I, int E, int k, int n_sm)
{
    if (n_sm > kMaxGridCtas) return false;
    return fused_plan_for(H, I, E, k, n_sm).slots >= 2;
}

cudaError_t launch_decode1_fused(const void *x, const float *logits, const void *wgu, const void *wd, int H, int I,
                                 int E, int k, int n_sm, float *gu, unsigned long long *flags, int32_t *idx_out,
                                 float *w_out, float *out, cudaStream_t s)
{
    const FusedPlan p = fused_plan_for(H, I, E, k, n_sm);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_sm);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = layout(p.slots, p.slot_bytes, E, p.payload).total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode1_fused_kernel, (const uint16_t *)x, logits, (const uint16_t *)wgu,
                              (const uint16_t *)wd, H, I, E, k, p.slots, p.slot_bytes, p.rpc, p.rpd, p.nh_max, gu,
                              flags, next_epoch(), idx_out, w_out, out);
}

cudaError_t read_decode1_fault_word(uint32_t *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_decode1_fault_word, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_decode1_fault_word, &zero, sizeof(uint32_t));
}

cudaError_t decode1_init_device()
{
    for (const void *kern : {(const void *)decode1_gate_up_kernel, (const void *)decode1_down_kernel,
                             (const void *)decode1_fused_kernel}) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
        if (e == cudaSuccess)  // ask for the largest shared-memory carveout so both CTAs fit
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool decode1_supported(int H, int I, int E, int k, int n_sm)
{
    const Plan p = plan_for(H, I, E, k, n_sm);
    return p.slots_a >= 2 && p.slots_b >= 2;
}

cudaError_t launch_decode1(const void *x, const float *logits, const void *wgu, const void *wd, int H, int I, int E,
                           int k, int n_sm, float *gu, int32_t *idx_out, float *w_out, float *out, cudaStream_t s,
                           cudaEvent_t between)
{
    const Plan p = plan_for(H, I, E, k, n_sm);
    const size_t smem_a = layout(p.slots_a, p.rpc * 2 * H, E, p.payload_a).total;
    decode1_gate_up_kernel<<<n_sm, kThreads, smem_a, s>>>((const uint16_t *)x, logits, (const uint16_t *)wgu, H, I,
                                                          E, k, p.slots_a, p.rpc, gu, idx_out, w_out);
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    if (between) {
        e = cudaEventRecord(between, s);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_sm);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = layout(p.slots_b, p.rpd * 2 * I, E, p.payload_b).total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode1_down_kernel, (const float *)gu, logits, (const uint16_t *)wd, H, I, E, k,
                              p.slots_b, p.rpd, p.nh_max, out);
}

}  // namespace moe
