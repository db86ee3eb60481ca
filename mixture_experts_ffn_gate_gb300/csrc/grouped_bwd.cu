// grouped_bwd.cu -- the backward pass's own kernels: the sorted-row inputs,
// the weight gradients on the tensor cores and the router-logit gradient.
//
// The Mixture-of-Kittens article (section 2.37배는 어떤 기준선과 비교한
// 숫자인가) measures the MoE layer's backward pass in training; its
// gradients are the chain rule of the forward layer:
//   q = W_down[e]^T dout_t,  dw_j = act . q,  da = w q,
//   dg = da u s (1 + g (1 - s)),  du = da g s       (s = sigmoid(g)),
//   dx_t = sum_j (W_gate[e]^T dg + W_up[e]^T du),
//   dW_down[e] = sum_r (w dout_t) act^T,  dW_gate_up[e] = sum_r [dg ; du] x_t^T,
//   dlogits[t, s_j] = w_j (dw_j - sum_m w_m dw_m).
// The q and dx GEMMs run in grouped_gemm.cu (the weight rows on the MMA's M
// side, read along their other axis).  Here:
//
//   bwd_prep_kernel  -- per row r of the padded sorted order (each expert's
//     segment rounded up to 16 rows): x_s[r] = x[t] (BF16), dout split into
//     a BF16 pair ds_hi[r] + ds_lo[r] (~16 significant bits, the
//     split-precision products of Markidis et al. 2018, "NVIDIA Tensor Core
//     Programmability, Performance & Precision") and the routing weight
//     w_s[r]; pad rows are zeros.
//   wgrad_kernel     -- dW[e] [M x N] = sum over e's rows of A[r] (x) B[r]:
//       dW_down:    A = ds_hi/lo [rows][H],   B = wa_hi/lo [rows][I]
//                   (hi.hi + hi.lo + lo.hi: the lo.lo term is below 2^-16
//                   of the product)
//       dW_gate_up: A = dgu_hi/lo [rows][2I], B = x_s [rows][H]
//                   (hi.x + lo.x; x is exact in BF16)
//     One item is one 128 x 256 output tile of one expert; K is the
//     expert's rows in steps of 32 (the MMA's K steps of 16 stop at the
//     16-row padding, whose rows are zero).  Both operands are MN-major:
//     TMA boxes of 64 elements (128 bytes, 128-byte swizzle) by 32 rows.
//     Experts without rows are skipped: zero_untouched_kernel has written
//     their zeros with plain 16-byte stores.  Each output element is one MMA
//     chain in a fixed order, so the gradients are bit-identical from run
//     to run whatever the grid.
//   zero_untouched_kernel -- the gradients of the experts no row selects,
//     written as zeros by a plain write stream before the weight-gradient
//     kernels run (they skip those experts).
//   dlogits_kernel   -- one warp per token: dw_j from the q epilogue's
//     partial sums (fixed order), then the softmax gradient.
//
// One persistent CTA per SM runs wgrad: warp 0 issues the TMA loads into
// a ring of stages, warp 1 the MMAs into one of two 256-column TMEM
// accumulators, warps 2-9 drain the other one (two warps per TMEM lane
// quarter, 128 columns each).  The gradients are written by TMA tensor
// stores: each epilogue warp places a 32-row x 32-column FP32 block in its
// 128-byte-swizzled staging buffer and hands it to the TMA engine, so every
// row leaves as one 128-byte line (a warp's own stores, one row per lane,
// would split into 32 partial sectors).  Every mbarrier
// wait is bounded; on time-out the CTA raises a bit in the device fault
// word, drains what it has in flight (bounded) and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace moe {

// the weight-gradient kernels' fault bits (FAULT_GEMM_*), read and cleared
// with the other kernels' words
__device__ uint32_t g_bwd_fault_word = 0;

cudaError_t read_bwd_fault_word(uint32_t *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_bwd_fault_word, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_bwd_fault_word, &zero, sizeof(uint32_t));
}

namespace {

constexpr int WBM = 128;               // output rows per tile (MMA M)
constexpr int WNB = 256;               // output columns per tile (MMA N)
constexpr int WK = 32;                 // rows per K step (TMA box height)
constexpr int BOX = 64 * WK * 2;       // one 64-element x 32-row BF16 box: 4 KB
constexpr int kWThreads = 320;         // producer, MMA issuer, 8 epilogue warps
constexpr int kEpiWarps = 8;
constexpr int OUT_BLOCK = 32 * 32 * 4;  // one staged 32 x 32 FP32 output block: 4 KB
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;

enum : int { kDwDown = 0, kDwGateUp = 1 };

template <int KIND>
struct WCfg {
    static constexpr bool B_PAIR = KIND == kDwDown;      // B is a hi/lo pair (wa); else x_s
    static constexpr int A_HALF = (WBM / 64) * BOX;      // 16 KB: the tile's rows of A_hi (or A_lo)
    static constexpr int B_HALF = (WNB / 64) * BOX;      // 32 KB
    static constexpr int A_BYTES = 2 * A_HALF;
    static constexpr int B_BYTES = (B_PAIR ? 2 : 1) * B_HALF;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = B_PAIR ? 4 : 5;
    // one staged block per epilogue warp: the shared memory serves the
    // operand stages better (measured: two blocks per warp and one stage
    // fewer, 2.62 / 5.00 ms at T = 2048; one block, 2.53 / 4.92 ms)
    static constexpr int STAGING = kEpiWarps * OUT_BLOCK;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + STAGING + 256;
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct WArgs {
    const int32_t *offs;    // [E+1] padded segment starts
    const int32_t *counts;  // [E] rows per expert
    int M, N, E;            // output [E][M][N] (written through the output tensor map)
    int m_tiles, n_tiles;
};

__device__ __forceinline__ void raise(uint32_t bit) { atomicOr(&g_bwd_fault_word, bit); }

template <int KIND>
__global__ void __launch_bounds__(kWThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                 const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                 const __grid_constant__ CUtensorMap tmOut, const WArgs args)
{
    // tmOut: the gradient [E][M][N] FP32, box 32 x 32 x 1, 128-byte swizzle
    using C = WCfg<KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *staging = smem + C::STAGES * C::STAGE_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(staging + C::STAGING);
    uint64_t *empty = full + C::STAGES;
    uint64_t *tfull = empty + C::STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull + b, 1);
            ptx::mbar_init(tempty + b, 8);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tmAh);
        ptx::prefetch_tensormap(&tmAl);
        ptx::prefetch_tensormap(&tmBh);
        if (C::B_PAIR) ptx::prefetch_tensormap(&tmBl);
        ptx::prefetch_tensormap(&tmOut);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, 2 * WNB);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int per_e = args.m_tiles * args.n_tiles;
    const int total = args.E * per_e;
    // item i: expert i / per_e, then output row tile, then column tile
    auto decode = [&](int i, int &e, int &m0, int &n0, int &rows, int &r0) {
        e = i / per_e;
        const int rem = i - e * per_e;
        const int mt = rem / args.n_tiles;
        m0 = mt * WBM;
        n0 = (rem - mt * args.n_tiles) * WNB;
        rows = __ldg(args.counts + e);
        r0 = __ldg(args.offs + e);
    };

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[C::STAGES];
            for (int s = 0; s < C::STAGES; ++s) armed[s] = 0;
            for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x) {
                int e, m0, n0, rows, r0;
                decode(i, e, m0, n0, rows, r0);
                for (int kr = 0; kr < rows; kr += WK) {
                    if (!ptx::mbar_wait_bounded(empty + stage, phase ^ 1, abort_flag, kWaitNs)) {
                        if (!*abort_flag) raise(FAULT_GEMM_PRODUCER);
                        *abort_flag = 1;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(full + stage, C::STAGE_BYTES);
                    ++armed[stage];
                    uint8_t *a = smem + stage * C::STAGE_BYTES;
                    uint8_t *b = a + C::A_BYTES;
                    const int r = r0 + kr;
#pragma unroll
                    for (int h = 0; h < WBM / 64; ++h) {
                        ptx::tma_load_2d(a + h * BOX, &tmAh, m0 + 64 * h, r, full + stage);
                        ptx::tma_load_2d(a + C::A_HALF + h * BOX, &tmAl, m0 + 64 * h, r, full + stage);
                    }
#pragma unroll
                    for (int h = 0; h < WNB / 64; ++h) {
                        ptx::tma_load_2d(b + h * BOX, &tmBh, n0 + 64 * h, r, full + stage);
                        if (C::B_PAIR) ptx::tma_load_2d(b + C::B_HALF + h * BOX, &tmBl, n0 + 64 * h, r, full + stage);
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            const volatile int keep_waiting = 0;
            for (int s = 0; s < C::STAGES; ++s)
                if (armed[s]) ptx::mbar_wait_bounded(full + s, (armed[s] - 1) & 1, &keep_waiting, kDrainNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int li = 0;  // items with rows, in this CTA's order
            const uint32_t idesc = ptx::idesc_bf16_f32_mn(WBM, WNB, true, true);
            for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x) {
                int e, m0, n0, rows, r0;
                decode(i, e, m0, n0, rows, r0);
                if (rows == 0) continue;
                const int acc = li & 1;
                const uint32_t aph = (li >> 1) & 1;
                ++li;
                if (!ptx::mbar_wait_bounded(tempty + acc, aph ^ 1, abort_flag, kWaitNs)) {
                    if (!*abort_flag) raise(FAULT_GEMM_MMA);
                    *abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * WNB;
                const int padded = (rows + 15) & ~15;
                bool ok = true;
                for (int kr = 0; kr < rows; kr += WK) {
                    if (!ptx::mbar_wait_bounded(full + stage, phase, abort_flag, kWaitNs)) {
                        if (!*abort_flag) raise(FAULT_GEMM_MMA);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
                    const int nk = min(WK, padded - kr) / 16;   // 1 or 2
                    for (int k = 0; k < nk; ++k) {
                        const uint64_t ah = ptx::sw128_desc_mn(a_addr + k * 2048, BOX);
                        const uint64_t al = ptx::sw128_desc_mn(a_addr + C::A_HALF + k * 2048, BOX);
                        const uint64_t bh = ptx::sw128_desc_mn(b_addr + k * 2048, BOX);
                        ptx::mma_bf16(d, ah, bh, idesc, (kr | k) != 0);
                        if (C::B_PAIR) {
                            const uint64_t bl = ptx::sw128_desc_mn(b_addr + C::B_HALF + k * 2048, BOX);
                            ptx::mma_bf16(d, ah, bl, idesc, 1);
                        }
                        ptx::mma_bf16(d, al, bh, idesc, 1);
                    }
                    ptx::mma_commit(empty + stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(tfull + acc);
            }
            ptx::mma_commit(drain);
            ptx::mbar_wait_bounded(drain, 0, abort_flag, kDrainNs);
        }
    } else {
        // ---------------------------------------------------- epilogue
        // warps 2..9: TMEM lane quarter warp % 4 (output rows m0 + 32 q ..),
        // columns half * 128 ... in four 32-column blocks.  Lane l holds row
        // l of a block; its 16-byte piece j goes to (j ^ (l % 8)) * 16 of the
        // row's 128 bytes in the staging buffer (the tensor map's swizzle).
        const int q = warp & 3, half = (warp - 2) >> 2;
        uint8_t *stg = staging + (warp - 2) * OUT_BLOCK;
        auto put_block = [&](const uint32_t (&r)[32], int e, int row0, int col0) {
            uint8_t *b = stg + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4 *>(b + ((j ^ (lane & 7)) << 4)) =
                    make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // rows past M and columns past N are not written by the store
                ptx::tma_store_3d(&tmOut, stg, col0, row0, e);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_read<0>();   // the buffer is free again once the store has read it
            }
            __syncwarp();
        };
        int li = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x) {
            int e, m0, n0, rows, r0;
            decode(i, e, m0, n0, rows, r0);
            const int row0 = m0 + 32 * q;
            const bool rows_in = row0 < args.M;   // M is a multiple of 32: a block is all in or all out
            if (rows == 0) continue;   // nothing selected this expert: zero_untouched_kernel wrote its zeros
            const int acc = li & 1;
            const uint32_t aph = (li >> 1) & 1;
            ++li;
            if (*abort_flag || !ptx::mbar_wait_bounded(tfull + acc, aph, abort_flag, kWaitNs)) {
                if (!*abort_flag) raise(FAULT_GEMM_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + acc * WNB;
            for (int c0 = half * (WNB / 2); c0 < (half + 1) * (WNB / 2); c0 += 32) {
                uint32_t r[32];
                ptx::tmem_ld32(tbase + c0, r);
                ptx::tmem_wait_ld();
                // N is a multiple of 64, so a 32-column block is all in or all out
                if (rows_in && n0 + c0 < args.N) put_block(r, e, row0, n0 + c0);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty + acc);
        }
        if (lane == 0) ptx::bulk_wait_all();   // the last stores have left shared memory and landed
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, 2 * WNB);
}

// ---------------------------------------------------------------- prep
// Block per padded row (grid-stride): the row's token, dout split, weight.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t *__restrict__ x,
                                                       const float *__restrict__ dout, const float *__restrict__ w,
                                                       const int32_t *__restrict__ perm,
                                                       const int32_t *__restrict__ offs, int E, int H, int k,
                                                       uint16_t *__restrict__ xs, __nv_bfloat16 *__restrict__ ds_hi,
                                                       __nv_bfloat16 *__restrict__ ds_lo, float *__restrict__ w_s)
{
    const int n_rows = __ldg(offs + E);
    for (int r = blockIdx.x; r < n_rows; r += gridDim.x) {
        const int a = __ldg(perm + r);
        const int t = a >= 0 ? a / k : 0;
        if (threadIdx.x == 0) w_s[r] = a >= 0 ? __ldg(w + a) : 0.0f;
        // 8 elements per step: 16 bytes of x, 32 bytes of dout
        for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
            uint4 xv = make_uint4(0, 0, 0, 0);
            float d[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (a >= 0) {
                xv = __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)t * H) + c);
                const float4 d0 = __ldg(reinterpret_cast<const float4 *>(dout + (int64_t)t * H) + 2 * c);
                const float4 d1 = __ldg(reinterpret_cast<const float4 *>(dout + (int64_t)t * H) + 2 * c + 1);
                d[0] = d0.x, d[1] = d0.y, d[2] = d0.z, d[3] = d0.w;
                d[4] = d1.x, d[5] = d1.y, d[6] = d1.z, d[7] = d1.w;
            }
            reinterpret_cast<uint4 *>(xs + (int64_t)r * H)[c] = xv;
            __align__(16) __nv_bfloat16 hi[8], lo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                hi[j] = __float2bfloat16_rn(d[j]);
                lo[j] = __float2bfloat16_rn(d[j] - __bfloat162float(hi[j]));
            }
            reinterpret_cast<uint4 *>(ds_hi + (int64_t)r * H)[c] = *reinterpret_cast<const uint4 *>(hi);
            reinterpret_cast<uint4 *>(ds_lo + (int64_t)r * H)[c] = *reinterpret_cast<const uint4 *>(lo);
        }
    }
}

// ---------------------------------------------------------------- zeros
// The weight gradients of the experts no row selects are zero: every block
// walks the experts in order and, for each one with counts[e] == 0, writes
// its share of dW_gate_up[e] and dW_down[e] with 16-byte stores (four
// whole 128-byte lines per warp instruction, a plain write stream).
__global__ void __launch_bounds__(256) zero_untouched_kernel(const int32_t *__restrict__ counts, int E,
                                                             float4 *__restrict__ dwgu, int64_t gu4,
                                                             float4 *__restrict__ dwd, int64_t d4)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fill = [&](float4 *p, int64_t n) {
        int64_t i = first;
        for (; i + 3 * stride < n; i += 4 * stride) {   // four independent stores per step
            p[i] = z;
            p[i + stride] = z;
            p[i + 2 * stride] = z;
            p[i + 3 * stride] = z;
        }
        for (; i < n; i += stride) p[i] = z;
    };
    for (int e = 0; e < E; ++e) {
        if (__ldg(counts + e) != 0) continue;
        fill(dwgu + (int64_t)e * gu4, gu4);
        fill(dwd + (int64_t)e * d4, d4);
    }
}

// ---------------------------------------------------------------- dlogits
// One warp per token: dw_j = sum_g dwp[pos][g] (g ascending), S = sum_j w_j
// dw_j (j ascending), dlogits[t, idx_j] = w_j (dw_j - S), zero elsewhere.
__global__ void __launch_bounds__(256) dlogits_kernel(const float *__restrict__ dwp, const int32_t *__restrict__ pos,
                                                      const int32_t *__restrict__ idx, const float *__restrict__ w,
                                                      int T, int E, int k, int groups, float *__restrict__ dlogits)
{
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    float *row = dlogits + (int64_t)t * E;
    for (int e = lane; e < E; e += 32) row[e] = 0.0f;
    // k <= 32: lane j owns slot j
    float dw = 0.0f, wj = 0.0f;
    int ej = 0;
    if (lane < k) {
        const int64_t a = (int64_t)t * k + lane;
        const float *p = dwp + (int64_t)__ldg(pos + a) * groups;
        for (int g = 0; g < groups; ++g) dw += __ldg(p + g);
        wj = __ldg(w + a);
        ej = __ldg(idx + a);
    }
    float S = 0.0f;
    for (int j = 0; j < k; ++j) S = fmaf(__shfl_sync(0xffffffffu, wj, j), __shfl_sync(0xffffffffu, dw, j), S);
    __syncwarp();
    if (lane < k) row[ej] = wj * (dw - S);
}

template <int KIND>
cudaError_t set_wgrad_smem()
{
    return cudaFuncSetAttribute(wgrad_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, WCfg<KIND>::SMEM);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn wencoder()
{
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// [rows][cols] BF16, box 64 columns (128 bytes, 128-byte swizzle) x 64 rows
cudaError_t make_rows_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols)
{
    EncodeTiledFn enc = wencoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, WK};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// the gradient [E][M][N] FP32, box 32 columns (128 bytes, 128-byte swizzle)
// x 32 rows x 1 expert
cudaError_t make_out_map(CUtensorMap *map, float *base, uint64_t E, uint64_t M, uint64_t N)
{
    EncodeTiledFn enc = wencoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {N, M, E};
    const cuuint64_t strides[2] = {N * 4, N * M * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int KIND>
cudaError_t launch_wgrad(const void *ah, const void *al, const void *bh, const void *bl, const int32_t *offs,
                         const int32_t *counts, int n_rows, int M, int N, int E, float *out, int ctas, cudaStream_t s)
{
    CUtensorMap tAh, tAl, tBh, tBl, tOut;
    cudaError_t e = make_rows_map(&tAh, ah, n_rows, M);
    if (e == cudaSuccess) e = make_rows_map(&tAl, al, n_rows, M);
    if (e == cudaSuccess) e = make_rows_map(&tBh, bh, n_rows, N);
    if (e == cudaSuccess) e = make_rows_map(&tBl, bl ? bl : bh, n_rows, N);
    if (e == cudaSuccess) e = make_out_map(&tOut, out, E, M, N);
    if (e != cudaSuccess) return e;
    const WArgs a{offs, counts, M, N, E, (M + WBM - 1) / WBM, (N + WNB - 1) / WNB};
    const int64_t items = (int64_t)E * a.m_tiles * a.n_tiles;
    const int grid = (int)(items < ctas ? items : ctas);
    wgrad_kernel<KIND><<<grid, kWThreads, WCfg<KIND>::SMEM, s>>>(tAh, tAl, tBh, tBl, tOut, a);
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t bwd_init_device()
{
    cudaError_t e = set_wgrad_smem<kDwDown>();
    if (e == cudaSuccess) e = set_wgrad_smem<kDwGateUp>();
    return e;
}

cudaError_t launch_bwd_prep(const void *x, const float *dout, const float *w, const int32_t *perm,
                            const int32_t *offs, int n_rows_max, int E, int H, int k, void *xs, void *ds_hi,
                            void *ds_lo, float *w_s, int n_sm, cudaStream_t s)
{
    const int grid = n_rows_max < 8 * n_sm ? (n_rows_max > 0 ? n_rows_max : 1) : 8 * n_sm;
    bwd_prep_kernel<<<grid, 256, 0, s>>>((const uint16_t *)x, dout, w, perm, offs, E, H, k, (uint16_t *)xs,
                                         (__nv_bfloat16 *)ds_hi, (__nv_bfloat16 *)ds_lo, w_s);
    return cudaPeekAtLastError();
}

cudaError_t launch_wgrad_down(const void *ds_hi, const void *ds_lo, const void *wa_hi, const void *wa_lo,
                              const int32_t *offs, const int32_t *counts, int n_rows, int H, int I, int E,
                              float *dwd, int ctas, cudaStream_t s)
{
    return launch_wgrad<kDwDown>(ds_hi, ds_lo, wa_hi, wa_lo, offs, counts, n_rows, H, I, E, dwd, ctas, s);
}

cudaError_t launch_wgrad_gate_up(const void *dgu_hi, const void *dgu_lo, const void *xs, const int32_t *offs,
                                 const int32_t *counts, int n_rows, int H, int I, int E, float *dwgu, int ctas,
                                 cudaStream_t s)
{
    return launch_wgrad<kDwGateUp>(dgu_hi, dgu_lo, xs, nullptr, offs, counts, n_rows, 2 * I, H, E, dwgu, ctas, s);
}

cudaError_t launch_zero_untouched(const int32_t *counts, int E, int H, int I, float *dwgu, float *dwd, int n_sm,
                                  cudaStream_t s)
{
    // 2I*H and H*I are multiples of 4 (H and I are multiples of 64)
    zero_untouched_kernel<<<8 * n_sm, 256, 0, s>>>(counts, E, reinterpret_cast<float4 *>(dwgu),
                                                   (int64_t)2 * I * H / 4, reinterpret_cast<float4 *>(dwd),
                                                   (int64_t)H * I / 4);
    return cudaPeekAtLastError();
}

cudaError_t launch_dlogits(const float *dwp, const int32_t *pos, const int32_t *idx, const float *w, int T, int E,
                           int k, int I, float *dlogits, cudaStream_t s)
{
    dlogits_kernel<<<(unsigned)ceil_div(T, 8), 256, 0, s>>>(dwp, pos, idx, w, T, E, k, I / 32, dlogits);
    return cudaPeekAtLastError();
}

}  // namespace moe
