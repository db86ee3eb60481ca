// grouped_gemm.cu -- the large-T path's grouped GEMMs on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// Large batches are the regime where grouping tokens by expert pays (the
// warp-decode article, section 배경 및 맥락, calls expert-grouped MoE efficient
// for training and large batches, and section 경쟁 구도 / 비교 treats prefill
// and decode as different problems).  After the counting sort, the tokens of
// expert e are rows [offs[e], offs[e+1]) of the sorted order, cut into chunks
// of at most kGemmChunkMax rows.
//
// Both GEMMs put the expert's weight rows on the MMA's M side (M = 128) and
// the chunk's tokens on the N side (N = chunk rounded up to 16, <= 64), so
// a skewed or tiny expert load never pads the weight tile.  A work item is
// one chunk against MT weight tiles of one expert (gate_up 4, down 3), which
// share the chunk's token tile:
//   gate_up: D[128 x N] = W_gu[e][rows] . x[tokens of the chunk]^T, K = H.
//            The chunk's token rows are read from x by the sorted order (row
//            p is token perm[p] / k), so no gathered copy of x is built.
//            The 128 rows of
//            a tile are 4 groups of (16 gate rows i.., 16 up rows I+i..), so
//            each epilogue warp holds gate and up of the same 16 neurons in
//            its lanes 0-15 / 16-31 and pairs them with one shuffle.  The
//            epilogue writes act = silu(g)*u as an unevaluated BF16 pair
//            hi = bf16(act), lo = bf16(act - hi), keeping ~16 significant
//            bits of the FP32 intermediate for the down GEMM (split-precision
//            products as in Markidis et al. 2018, "NVIDIA Tensor Core
//            Programmability, Performance & Precision").
//   down:    D[128 x N] = W_down[e][h0:h0+128] . [act_hi ; act_lo][chunk]^T,
//            K = I: the chunk's hi rows and then its lo rows form one B tile,
//            so one MMA per K step reads the weight tile once for both halves
//            (with a few tokens on N the tensor pipe's time goes into reading
//            the 128 x 16 weight slice from shared memory, so a second MMA
//            for the lo half would cost as much as the first); the epilogue
//            writes z[sorted row, h] = D[:, j] + D[:, box + j] in FP32.
// Every output element is one MMA chain over K in a fixed order, so results
// do not depend on the grid size or on which CTA ran which tile.
//
// One persistent CTA per SM: warp 0 issues TMA loads into a ring of smem
// stages, warp 1 issues tcgen05.mma into one of two TMEM accumulators,
// warps 2-5 drain the other accumulator (tcgen05.ld) and store.  gate_up
// has three more warps, one per ring stage, that copy the chunk's x rows
// into their stage (16-byte cp.async copies placed at the 128-byte-swizzled
// offsets the MMA's B descriptor expects), wait for them, fence the proxies
// and give the stage's full barrier its second arrival.  Every
// mbarrier wait is bounded: on time-out the CTA raises a bit in the device
// fault word, lets its copies and MMAs in flight finish (again bounded),
// frees its TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace moe {

__device__ uint32_t g_fault_word = 0;

__device__ __forceinline__ void raise_fault(uint32_t bit) { atomicOr(&g_fault_word, bit); }

cudaError_t read_fault_word(uint32_t *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_fault_word, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(uint32_t));
}

namespace {

constexpr int BM = 128;                  // weight rows per tile (MMA M)
constexpr int BK = 64;                   // K elements per stage: one 128-byte swizzle row
constexpr int NMAX = kGemmChunkMax;      // tokens per chunk (MMA N <= NMAX)
constexpr int ACC_COLS = 64;             // TMEM columns per accumulator (>= NMAX)
constexpr int SMALL_ROWS = 16;           // B box for chunks of at most 16 rows
constexpr int kThreads = 192;           // down: producer, MMA issuer, 4 epilogue warps
constexpr int kThreadsGateUp = 288;     // gate_up: + one x-row loader warp per ring stage
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr int kPrefetchSteps = 6;                 // MX: code boxes fetched into L2 this far ahead
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s to drain after an abort

static_assert(NMAX <= ACC_COLS && NMAX % 16 == 0, "chunk must fit one accumulator");

// What a kernel instance computes (the forward pass's two GEMMs, and the
// backward pass's recomputation of gate/up and its two GEMMs against the
// weights read along their other axis).
enum : int {
    kDown = 0,       // z = W_down . [act_hi ; act_lo]
    kGateUp = 1,     // act = silu(W_gate x) * (W_up x) as a BF16 hi/lo pair
    kGateUpRaw = 2,  // g = W_gate x and u = W_up x in FP32
    kBwdQ = 3,       // q = W_down^T . [dout_hi ; dout_lo], then the SwiGLU backward
    kBwdDx = 4,      // z = W_gate_up^T . [dgu_hi ; dgu_lo]
    kGateUpMx = 5,   // kGateUp with MXFP8 weights
    kDownMx = 6,     // kDown with MXFP8 weights
    kGateUpSave = 7, // kGateUp that also keeps g and u in FP32 (the training forward)
};

template <int KIND>
struct Cfg {
    // MXFP8 weights: the producer loads E4M3 code tiles, converter warps
    // write them as exact BF16 (each 32-element block times its E8M0
    // scale) into the tile the MMA reads
    static constexpr bool MX = KIND == kGateUpMx || KIND == kDownMx;
    static constexpr bool GATE_UP = KIND == kGateUp || KIND == kGateUpRaw || KIND == kGateUpMx || KIND == kGateUpSave;
    // the weight tile is read along its rows' index (MN-major): the
    // backward's contractions over H (W_down) and over 2I (W_gate_up)
    static constexpr bool A_MN = KIND == kBwdQ || KIND == kBwdDx;
    // epilogue warps: q's SwiGLU backward reads and writes several arrays
    // per element, so two warps share each TMEM lane quarter (one 32-column
    // block each) to drain its single accumulator set sooner
    static constexpr int EPI_WARPS = KIND == kBwdQ ? 8 : 4;
    static constexpr int CONV_WARPS = MX ? 8 : 0;
    static constexpr int FIRST_CONV = 2 + EPI_WARPS + (GATE_UP ? 3 : 0);  // after the x-row loaders
    static constexpr int THREADS = 32 * (FIRST_CONV + CONV_WARPS);
    // weight tiles per item (they share one token tile); q takes two, so
    // that its accumulators fit twice (its long epilogue then overlaps the
    // next item's MMAs) and I's 128-row tiles split evenly
    // (MX: two, so that the code tiles fit beside three stages)
    static constexpr int MT = MX ? 2 : GATE_UP ? 4 : KIND == kBwdQ ? 2 : 3;
    // accumulator columns per weight tile: the chunk's tokens (gate_up), or
    // its hi rows then its lo rows (down, q, dx); gate_up and q double-buffer
    // them so the epilogue of one item overlaps the MMAs of the next, down
    // and dx (three tiles of 128 columns) have room for one set
    static constexpr int TILE_COLS = GATE_UP ? ACC_COLS : 2 * ACC_COLS;
    static constexpr int ACC_BUFS = GATE_UP || KIND == kBwdQ || MX ? 2 : 1;
    static constexpr int TMEM_COLS = ACC_BUFS * MT * TILE_COLS;
    // tcgen05.alloc takes a power of two of at least 32 columns
    static constexpr int TMEM_ALLOC = TMEM_COLS <= 32    ? 32
                                      : TMEM_COLS <= 64  ? 64
                                      : TMEM_COLS <= 128 ? 128
                                      : TMEM_COLS <= 256 ? 256
                                                         : 512;
    static_assert(TMEM_COLS <= 512, "accumulators exceed TMEM");
    static constexpr int STAGES = KIND == kBwdQ ? 4 : 3;
    static constexpr int A_TILE = BM * BK * 2;                            // 16 KB per weight tile
    static constexpr int A_BYTES = MT * A_TILE;
    static constexpr int B_TILE = NMAX * BK * 2;                          // 8 KB per operand
    static constexpr int B_BYTES = B_TILE * (GATE_UP ? 1 : 2);            // x | act_hi + act_lo
    static constexpr int CODE_TILE = BM * BK;                             // 8 KB of E4M3 codes per tile
    static constexpr int CODE_BYTES = MX ? MT * CODE_TILE : 0;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + CODE_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(THREADS == (GATE_UP && !MX ? kThreadsGateUp : THREADS), "gate_up keeps 288 threads");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Inputs and outputs of the backward pass's q GEMM epilogue (kBwdQ), all
// indexed by the (padded) sorted row r: g, u [rows][I] FP32 and the routing
// weight w_s [rows] in; dgu_hi/lo [rows][2I] (dg | du), wa_hi/lo [rows][I]
// (w * act) as BF16 pairs and dwp [rows][I/32] (partial sums of act . q
// over 32 neurons) out.
struct BwdQArgs {
    const float *g, *u, *w_s;
    __nv_bfloat16 *dgu_hi, *dgu_lo, *wa_hi, *wa_lo;
    float *dwp;
};

struct GemmArgs {
    const int4 *chunks;   // {expert, first sorted row, rows, first chunk of expert}
    const int32_t *nchunks;
    const int32_t *offs;  // [E+1] sorted-row offsets per expert
    int H, I;
    int K;                // reduction length (H or I)
    int m_tiles;          // groups of MT weight tiles per expert
    int tiles;            // weight tiles per expert (the last group may have fewer)
    int a_bytes;          // bytes of one weight box (MT tiles, fewer if the tensor is smaller)
    void *out0, *out1;    // act_hi, act_lo | z
    const uint16_t *x;    // gate_up: the tokens [T, H] (BF16 bits) and the
    const int32_t *perm;  // sorted order (assignment t*k+j at row p)
    int k;
    BwdQArgs q;           // kBwdQ only
    const uint8_t *scales;  // MX: the E8M0 scales [E][rows][scale_row] of the weight
    int scale_row;          // bytes per scale row (K / 32 padded to 16)
    float *g_keep, *u_keep; // kGateUpSave: g and u [rows][I] FP32 besides act
};

struct Item {
    int e, p0, n, m;      // m: group of MT weight tiles, tiles MT*m ... MT*m+MT-1
};

// Item i of the flat list: experts in order; within an expert, weight tile
// group m major and chunk minor, so the chunks that reuse one weight tile
// are adjacent (they run at about the same time and share it through L2).
__device__ __forceinline__ Item decode_item(int i, const GemmArgs &a)
{
    const int4 ch = __ldg(a.chunks + i / a.m_tiles);
    const int e = ch.x, c0 = ch.w;
    const int cnt = __ldg(a.offs + e + 1) - __ldg(a.offs + e);
    const int nc = (cnt + NMAX - 1) / NMAX;
    const int q = i - c0 * a.m_tiles;
    const int m = q / nc, c = c0 + (q - m * nc);
    const int4 cq = __ldg(a.chunks + c);
    return {e, cq.y, cq.z, m};
}

__device__ __forceinline__ int pad16(int n) { return (n + 15) & ~15; }

__device__ __forceinline__ void store_pair(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int64_t at, float v)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[at] = h;
    lo[at] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// After this, lane l holds the sum over the warp's 32 lanes of v[l] (a
// 32 x 32 transpose-and-add in 31 shuffles, in a fixed order): each round
// a lane keeps one half of its remaining columns and adds its partner's
// copy of that half.
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane)
{
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

// The backward pass's SwiGLU step for 32 columns (sorted rows it.p0 + c0 +
// j) of neuron i, whose q = W_down[e]^T dout_t values are r[j]:
//   s = sigmoid(g), a = g s u, da = w q,
//   dg = da u s (1 + g (1 - s)), du = da g s,
// stored as BF16 pairs (dgu rows: dg at i, du at I + i; wa = w a), zeros in
// the expert's pad rows; and act . q summed over the warp's 32 neurons
// into dwp[row][grp].
__device__ __forceinline__ void bwd_q_columns(const uint32_t (&r)[32], int ncols, int p0, int n, int c0, int i,
                                              int grp, const GemmArgs &args, int lane)
{
    const int I = args.I;
    const int npad = pad16(n);
    const BwdQArgs &b = args.q;
    float prod[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        // each half's loads first (predicated), so that they are in flight
        // together: the stores below could alias them as far as the
        // compiler knows, and would otherwise hold each column's loads back
        float gv[16], uv[16], wv[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int j = 16 * h + jj;
            const bool live = j < ncols && c0 + j < n;
            const int64_t row = p0 + c0 + j;
            gv[jj] = live ? __ldg(b.g + row * I + i) : 0.0f;
            uv[jj] = live ? __ldg(b.u + row * I + i) : 0.0f;
            wv[jj] = live ? __ldg(b.w_s + row) : 0.0f;
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int j = 16 * h + jj;
            const int col = c0 + j;
            prod[j] = 0.0f;
            if (j < ncols && col < npad) {
                const int64_t row = p0 + col;
                float dg = 0.0f, du = 0.0f, wa = 0.0f;
                if (col < n) {
                    const float qv = __uint_as_float(r[j]);
                    const float g = gv[jj], u = uv[jj], w = wv[jj];
                    const float sg = 1.0f / (1.0f + expf(-g));
                    const float silu = g * sg;
                    const float a = silu * u;
                    const float da = w * qv;
                    dg = da * u * (sg * (1.0f + g * (1.0f - sg)));
                    du = da * silu;
                    wa = w * a;
                    prod[j] = a * qv;
                }
                store_pair(b.dgu_hi, b.dgu_lo, row * 2 * I + i, dg);
                store_pair(b.dgu_hi, b.dgu_lo, row * 2 * I + I + i, du);
                store_pair(b.wa_hi, b.wa_lo, row * I + i, wa);
            }
        }
    }
    const float sum = warp_column_sums(prod, lane);
    if (lane < ncols && c0 + lane < n) b.dwp[(int64_t)(p0 + c0 + lane) * (I / 32) + grp] = sum;
}

template <int KIND>
__global__ void __launch_bounds__(Cfg<KIND>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0s,
                        const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1s,
                        const __grid_constant__ CUtensorMap tmB1, const GemmArgs args)
{
    // tmA: gate_up -- 5-D view of W_gu [E][2][I/16][16][H] (dims innermost
    //      first: H, 16 rows, gate|up, row group, expert) whose {64,16,2,4,1}
    //      box is one 128-row tile of 4 x (16 gate rows, 16 up rows);
    //      down -- 3-D [E][H][I], box 64 x 128 x 1 (one tile);
    //      q -- 3-D [E][H][I] with I innermost, box 64 (I) x 64 (H) x 1:
    //      two boxes (neurons i0.., i0+64..) per tile and K step;
    //      dx -- 3-D [E][2I][H] with H innermost, box 64 (H) x 64 (2I) x 1,
    //      two boxes (dims h0.., h0+64..) per tile and K step.
    // tmB0/tmB1 (down, q, dx): the chunk's hi/lo rows (act, dout or dgu),
    // box 64 x NMAX; tmB0s/tmB1s: the same with a 16-row box, for chunks of
    // <= 16 rows.  gate_up leaves the B maps unread.
    // MX (gate_up, down): tmA is the same view of the E4M3 codes (uint8,
    // no swizzle: 64-byte rows), its box a tile's codes.
    using C = Cfg<KIND>;
    constexpr bool GATE_UP = C::GATE_UP;
    constexpr bool A_MN = C::A_MN;
    constexpr bool MX = C::MX;
    constexpr int MT = C::MT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::STAGES * C::A_BYTES;
    uint8_t *sCode = sB + C::STAGES * C::B_BYTES;  // MX only
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *empty = full + C::STAGES;
    uint64_t *cfull = empty + C::STAGES;           // MX: a stage's codes (and down's B rows) landed
    uint64_t *tfull = cfull + C::STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // gate_up: the weight box's expect-tx arrival and the x rows'
            // arrival; MX: the converter warps' arrivals (and gate_up's x rows)
            ptx::mbar_init(full + s, MX ? C::CONV_WARPS + (GATE_UP ? 1 : 0) : GATE_UP ? 2 : 1);
            ptx::mbar_init(empty + s, 1);
            ptx::mbar_init(cfull + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull + b, 1);
            ptx::mbar_init(tempty + b, C::EPI_WARPS);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tmA);
        if (!GATE_UP) {
            ptx::prefetch_tensormap(&tmB0);
            ptx::prefetch_tensormap(&tmB0s);
            ptx::prefetch_tensormap(&tmB1);
            ptx::prefetch_tensormap(&tmB1s);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, C::TMEM_ALLOC);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int total = __ldg(args.nchunks) * args.m_tiles;
    const int KB = args.K / BK;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[C::STAGES];
            for (int s = 0; s < C::STAGES; ++s) armed[s] = 0;
            Item nxt = blockIdx.x < total ? decode_item(blockIdx.x, args) : Item{};
            for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x) {
                const Item it = nxt;
                if (i + (int)gridDim.x < total) nxt = decode_item(i + gridDim.x, args);  // loads overlap this item
                const bool small = it.n <= SMALL_ROWS;
                // gate_up: the weight box only (the x rows come from the loader warps)
                const uint32_t bytes = args.a_bytes + (GATE_UP ? 0 : (small ? SMALL_ROWS : NMAX) * BK * 2 * 2);
                uint64_t *const land = MX ? cfull : full;  // where the TMA copies complete
                for (int kb = 0; kb < KB; ++kb) {
                    if (!ptx::mbar_wait_bounded(empty + stage, phase ^ 1, abort_flag, kWaitLimitNs)) {
                        if (!*abort_flag) raise_fault(FAULT_GEMM_PRODUCER);
                        *abort_flag = 1;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(land + stage, bytes);
                    ++armed[stage];
                    const int k0 = kb * BK;
                    if constexpr (MX) {
                        // the code box kPrefetchSteps K steps on (this item's,
                        // or the next one's) into L2: a stage holds few code
                        // bytes, so its copies must not wait on DRAM
                        int pk = kb + kPrefetchSteps;
                        const Item *pi = &it;
                        if (pk >= KB) {
                            pk -= KB;
                            pi = (i + (int)gridDim.x < total && pk < KB) ? &nxt : nullptr;
                        }
                        if (pi) {
                            if (GATE_UP) {
                                ptx::tma_prefetch_5d(&tmA, pk * BK, 0, 0, pi->m * 4 * MT, pi->e);
                            } else {
#pragma unroll
                                for (int t = 0; t < MT; ++t)
                                    ptx::tma_prefetch_3d(&tmA, pk * BK, (pi->m * MT + t) * BM, pi->e);
                            }
                        }
                    }
                    uint8_t *a = MX ? sCode + stage * C::CODE_BYTES : sA + stage * C::A_BYTES;
                    // MT tiles: one box (gate_up) or one box per tile (down);
                    // rows past the expert's end read 0 and are never stored
                    if (GATE_UP) {
                        ptx::tma_load_5d(a, &tmA, k0, 0, 0, it.m * 4 * MT, it.e, land + stage);
                    } else if (MX) {
#pragma unroll
                        for (int t = 0; t < MT; ++t)
                            ptx::tma_load_3d(a + t * C::CODE_TILE, &tmA, k0, (it.m * MT + t) * BM, it.e, land + stage);
                    } else if (A_MN) {
#pragma unroll
                        for (int t = 0; t < MT; ++t) {
                            const int mn0 = (it.m * MT + t) * BM;
                            ptx::tma_load_3d(a + t * C::A_TILE, &tmA, mn0, k0, it.e, full + stage);
                            ptx::tma_load_3d(a + t * C::A_TILE + C::A_TILE / 2, &tmA, mn0 + 64, k0, it.e, full + stage);
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < MT; ++t)
                            ptx::tma_load_3d(a + t * C::A_TILE, &tmA, k0, (it.m * MT + t) * BM, it.e, full + stage);
                    }
                    // down: the hi rows, then the lo rows right after them (a
                    // whole number of 1024-byte swizzle groups), one B tile
                    if (!GATE_UP) {
                        uint8_t *b = sB + stage * C::B_BYTES;
                        ptx::tma_load_2d(b, small ? &tmB0s : &tmB0, k0, it.p0, land + stage);
                        ptx::tma_load_2d(b + (small ? SMALL_ROWS : NMAX) * BK * 2, small ? &tmB1s : &tmB1, k0, it.p0,
                                         land + stage);
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // let every armed copy land before the CTA can exit (the last
            // armed phase of each stage completes after all earlier ones)
            const volatile int keep_waiting = 0;
            for (int s = 0; s < C::STAGES; ++s)
                if (armed[s])
                    ptx::mbar_wait_bounded((MX ? cfull : full) + s, (armed[s] - 1) & 1, &keep_waiting, kDrainLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int li = 0;
            Item nxt = blockIdx.x < total ? decode_item(blockIdx.x, args) : Item{};
            for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x, ++li) {
                const Item it = nxt;
                if (i + (int)gridDim.x < total) nxt = decode_item(i + gridDim.x, args);
                // down: N spans the hi box and the lo rows that matter
                const int box = it.n <= SMALL_ROWS ? SMALL_ROWS : NMAX;
                const uint32_t idesc =
                    ptx::idesc_bf16_f32_mn(BM, GATE_UP ? pad16(it.n) : box + pad16(it.n), A_MN, false);
                const int acc = C::ACC_BUFS == 2 ? (li & 1) : 0;
                const uint32_t aph = C::ACC_BUFS == 2 ? (li >> 1) & 1 : li & 1;
                if (!ptx::mbar_wait_bounded(tempty + acc, aph ^ 1, abort_flag, kWaitLimitNs)) {
                    if (!*abort_flag) raise_fault(FAULT_GEMM_MMA);
                    *abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * MT * C::TILE_COLS;
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!ptx::mbar_wait_bounded(full + stage, phase, abort_flag, kWaitLimitNs)) {
                        if (!*abort_flag) raise_fault(FAULT_GEMM_MMA);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b_addr = ptx::smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t bd = ptx::sw128_desc(b_addr + k * 32);
#pragma unroll
                        for (int t = 0; t < MT; ++t) {
                            // K-major: the K step is 32 bytes along the row;
                            // MN-major: 16 K rows of 128 bytes, the tile's
                            // second 64-wide MN block a box (8 KB) on
                            const uint64_t ad = A_MN ? ptx::sw128_desc_mn(a_addr + t * C::A_TILE + k * 2048, C::A_TILE / 2)
                                                     : ptx::sw128_desc(a_addr + t * C::A_TILE + k * 32);
                            ptx::mma_bf16(d + t * C::TILE_COLS, ad, bd, idesc, (kb | k) != 0);
                        }
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
            // every MMA this thread issued has completed once drain fires
            ptx::mma_commit(drain);
            ptx::mbar_wait_bounded(drain, 0, abort_flag, kDrainLimitNs);
        }
    } else if (MX && warp >= C::FIRST_CONV) {
        // ------------------------------------ E4M3 -> BF16 converters (MX)
        // Per K step the stage holds MT tiles x 128 rows x 64 codes: 4
        // pieces of 16 codes per row, NP pieces per converter thread.  Piece
        // p = ct + NC j is chunk c = p & 3 of row r = (p >> 2) & 127 of tile
        // t = p >> 9; its 16 values, each code's value times the E8M0 scale
        // of its 32-element block (exact: the weights are BF16 numbers), go
        // to the row's 128-byte-swizzled 16-byte chunks 2c and 2c + 1.
        constexpr int NC = 32 * C::CONV_WARPS, NP = MT * BM * 4 / (NC > 0 ? NC : 1);
        static_assert(!MX || NP * NC == MT * BM * 4, "whole pieces per converter thread");
        const int ct = threadIdx.x - 32 * C::FIRST_CONV;
        // each piece's offsets in a stage's code buffer and BF16 tile
        uint32_t src_off[NP], dst_off0[NP], dst_off1[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const int p = ct + NC * j, c = p & 3, r = (p >> 2) & 127, t = p >> 9;
            src_off[j] = t * C::CODE_TILE + r * BK + c * 16;
            dst_off0[j] = t * C::A_TILE + r * 128 + (((2 * c) ^ (r & 7)) << 4);
            dst_off1[j] = t * C::A_TILE + r * 128 + (((2 * c + 1) ^ (r & 7)) << 4);
        }
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
            const Item it = decode_item(i, args);
            const uint8_t *srow[NP];  // each piece's scale row (null: a row past the weight's end)
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const int p = ct + NC * j, r = (p >> 2) & 127, t = p >> 9;
                int64_t grow;
                bool in;
                if constexpr (GATE_UP) {  // 4 groups x (16 gate rows, 16 up rows) of 16 neurons
                    const int neuron = ((it.m * MT + t) * 4 + (r >> 5)) * 16 + (r & 15);
                    in = neuron < args.I;
                    grow = ((int64_t)it.e * 2 + ((r >> 4) & 1)) * args.I + neuron;
                } else {
                    const int h = (it.m * MT + t) * BM + r;
                    in = h < args.H;
                    grow = (int64_t)it.e * args.H + h;
                }
                srow[j] = in ? args.scales + grow * args.scale_row : nullptr;
            }
            for (int kb = 0; kb < KB; ++kb) {
                uint32_t sc[NP];  // the scales do not depend on the codes: read them before the wait
#pragma unroll
                for (int j = 0; j < NP; ++j)
                    sc[j] = srow[j] ? __ldg(srow[j] + kb * 2 + (((ct + NC * j) & 3) >> 1)) : 127u;
                int got = 1;
                if (lane == 0) got = ptx::mbar_wait_bounded(cfull + stage, phase, abort_flag, kWaitLimitNs);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    if (lane == 0) {
                        if (!*abort_flag) raise_fault(FAULT_GEMM_CONVERT);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                const uint8_t *code = sCode + stage * C::CODE_BYTES;
                uint8_t *a = sA + stage * C::A_BYTES;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(code + src_off[j]);
                    const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
                    const float f = mx_f32_scale(sc[j]);
                    uint32_t w[8];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) e4m3x4_to_bf16x2_f32(cw[q2], f, w[2 * q2], w[2 * q2 + 1]);
                    *reinterpret_cast<uint4 *>(a + dst_off0[j]) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(a + dst_off1[j]) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                ptx::fence_proxy_async_smem();  // the MMA (async proxy) reads what these stores wrote
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(full + stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (GATE_UP && warp >= 6) {
        // ------------------------------------- x-row loaders (gate_up only)
        // Warp 6 + sl fills ring stage sl: the CTA's K steps n = sl, sl +
        // STAGES, ... over its items in the producer's order (item i = block
        // + j * grid, K steps in order; stage n % STAGES, phase (n / STAGES)
        // & 1).  Lane l copies rows l and l + 32 of the chunk, 128 bytes per
        // row, piece q of row r at (q ^ (r & 7)) * 16; rows past the chunk
        // are not loaded (the MMA's columns for them are never stored).
        const int sl = warp - 6;
        uint32_t swz[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) swz[q] = (uint32_t)((q ^ (lane & 7)) << 4);
        uint8_t *b = sB + sl * C::B_BYTES;
        int n = 0;  // this CTA's K steps before the current item
        for (int i = blockIdx.x; i < total; i += gridDim.x, n += KB) {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // warp-uniform
            // this item's K steps that fall on stage sl
            int kb = (sl - n % C::STAGES + C::STAGES) % C::STAGES;
            if (kb >= KB) continue;
            const Item it = decode_item(i, args);
            const uint16_t *row0 = nullptr, *row1 = nullptr;
            if (lane < it.n) row0 = args.x + (int64_t)(__ldg(args.perm + it.p0 + lane) / args.k) * args.H;
            if (lane + 32 < it.n) row1 = args.x + (int64_t)(__ldg(args.perm + it.p0 + lane + 32) / args.k) * args.H;
            bool ok = true;
            for (; kb < KB; kb += C::STAGES) {
                const uint32_t phase = (uint32_t)((n + kb) / C::STAGES) & 1u;
                int got = 1;
                if (lane == 0) got = ptx::mbar_wait_bounded(empty + sl, phase ^ 1, abort_flag, kWaitLimitNs);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    if (lane == 0) {
                        if (!*abort_flag) raise_fault(FAULT_GEMM_PRODUCER);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                const int k0 = kb * BK;
                if (row0) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) ptx::cp_async16(b + lane * 128 + swz[q], row0 + k0 + 8 * q);
                }
                if (row1) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) ptx::cp_async16(b + (lane + 32) * 128 + swz[q], row1 + k0 + 8 * q);
                }
                ptx::cp_async_commit();
                ptx::cp_async_wait_all();
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(full + sl);
            }
            if (!ok) break;
        }
        ptx::cp_async_wait_all();
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        // q: warps 2-5 take the chunk's 32-column blocks 0, 2, ..., warps 6-9 blocks 1, 3, ...
        const int c_first = C::EPI_WARPS == 8 ? 32 * ((warp - 2) >> 2) : 0;
        constexpr int c_step = C::EPI_WARPS == 8 ? 64 : 32;
        int li = 0;
        Item nxt = blockIdx.x < total ? decode_item(blockIdx.x, args) : Item{};
        for (int i = blockIdx.x; i < total; i += gridDim.x, ++li) {
            const Item it = nxt;
            if (i + (int)gridDim.x < total) nxt = decode_item(i + gridDim.x, args);
            const int acc = C::ACC_BUFS == 2 ? (li & 1) : 0;
            const uint32_t aph = C::ACC_BUFS == 2 ? (li >> 1) & 1 : li & 1;
            if (!ptx::mbar_wait_bounded(tfull + acc, aph, abort_flag, kWaitLimitNs)) {
                if (!*abort_flag) raise_fault(FAULT_GEMM_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            ptx::tc_fence_after();
            for (int t = 0; t < MT && it.m * MT + t < args.tiles; ++t) {
            const int tile = it.m * MT + t;
            // q: a warp whose 32 neurons lie past I has nothing to do
            if (KIND == kBwdQ && tile * BM + 32 * q >= args.I) continue;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + (acc * MT + t) * C::TILE_COLS;
            for (int c0 = c_first; c0 < it.n; c0 += c_step) {
                uint32_t r[32];
                ptx::tmem_ld32(tbase + c0, r);
                if (!GATE_UP) {
                    // z = hi part + lo part: for a small chunk both sit in
                    // these 32 columns (lo from column 16), else the lo part
                    // is 64 columns on
                    if (it.n > SMALL_ROWS) {
                        uint32_t rl[32];
                        ptx::tmem_ld32(tbase + NMAX + c0, rl);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(rl[j]));
                    } else {
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < SMALL_ROWS; ++j)
                            r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r[SMALL_ROWS + j]));
                    }
                } else {
                    ptx::tmem_wait_ld();
                }
                if constexpr (KIND == kGateUpRaw) {
                    const int neuron = tile * 64 + 16 * q + (lane & 15);
                    float *dst = reinterpret_cast<float *>(lane < 16 ? args.out0 : args.out1);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < it.n) dst[(int64_t)(it.p0 + c0 + j) * args.I + neuron] = __uint_as_float(r[j]);
                } else if constexpr (KIND == kBwdQ) {
                    bwd_q_columns(r, it.n > SMALL_ROWS ? 32 : SMALL_ROWS, it.p0, it.n, c0, tile * BM + 32 * q + lane,
                                  tile * 4 + q, args, lane);
                } else if constexpr (KIND == kGateUp || KIND == kGateUpMx || KIND == kGateUpSave) {
                    const int neuron = tile * 64 + 16 * q + (lane & 15);
                    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(lane < 16 ? args.out0 : args.out1);
                    float *keep = lane < 16 ? args.g_keep : args.u_keep;   // kGateUpSave: g (lanes 0-15), u
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float v = __uint_as_float(r[j]);
                        const float o = __shfl_xor_sync(0xffffffffu, v, 16);
                        const float a = lane < 16 ? swiglu(v, o) : swiglu(o, v);
                        const __nv_bfloat16 hi = __float2bfloat16_rn(a);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(a - __bfloat162float(hi));
                        if (c0 + j < it.n) {
                            const int64_t at = (int64_t)(it.p0 + c0 + j) * args.I + neuron;
                            dst[at] = lane < 16 ? hi : lo;
                            if constexpr (KIND == kGateUpSave) keep[at] = v;
                        }
                    }
                } else {
                    const int h = tile * BM + 32 * q + lane;
                    float *z = reinterpret_cast<float *>(args.out0);
                    if (h < args.H) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j < it.n) z[(int64_t)(it.p0 + c0 + j) * args.H + h] = __uint_as_float(r[j]);
                    }
                }
            }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty + acc);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, C::TMEM_ALLOC);
}

// ---------------------------------------------------------------- host
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder()
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

// A 2D BF16 tensor map over a row-major [rows, cols] matrix, box = 64 columns
// (128 bytes, 128-byte swizzle) x box_rows rows.  Rows past the end read 0.
cudaError_t make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// W_down [E, H, I] as a 3-D map (I, H, E), box 64 x 128 rows x 1 expert: one
// weight tile; rows past H read 0.
cudaError_t make_down_map(CUtensorMap *map, const void *base, int E, int H, int I)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)E};
    const cuuint64_t strides[2] = {(cuuint64_t)I * 2, (cuuint64_t)I * 2 * H};
    const cuuint32_t box[3] = {BK, BM, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// W_gate_up [E, 2I, H] viewed as [E][I/16][2][16][H] (dims innermost first:
// H, 16 rows, gate|up, group of 16 neurons, expert).  A {64, 16, 2, 4, 1}
// box at {k0, 0, 0, 4m, e} is neurons 64m..64m+63 of expert e laid out as
// 4 x (16 gate rows, 16 up rows), 128-byte swizzled.
cudaError_t make_gate_up_map(CUtensorMap *map, const void *base, int E, int I, int H, uint32_t groups)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t row = (cuuint64_t)H * 2;
    const cuuint64_t dims[5] = {(cuuint64_t)H, 16, 2, (cuuint64_t)I / 16, (cuuint64_t)E};
    const cuuint64_t strides[4] = {row, row * I, row * 16, row * 2 * I};
    const cuuint32_t box[5] = {BK, 16, 2, groups, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The same two weight views over MXFP8 codes (uint8 [E, 2I, H] and
// [E, H, I]): 64 codes (64 bytes) per box row, no swizzle.
cudaError_t make_gate_up_code_map(CUtensorMap *map, const void *base, int E, int I, int H, uint32_t groups)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t row = (cuuint64_t)H;
    const cuuint64_t dims[5] = {(cuuint64_t)H, 16, 2, (cuuint64_t)I / 16, (cuuint64_t)E};
    const cuuint64_t strides[4] = {row, row * I, row * 16, row * 2 * I};
    const cuuint32_t box[5] = {BK, 16, 2, groups, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_down_code_map(CUtensorMap *map, const void *base, int E, int H, int I)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)E};
    const cuuint64_t strides[2] = {(cuuint64_t)I, (cuuint64_t)I * H};
    const cuuint32_t box[3] = {BK, BM, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int grid_for(int ctas, int n_assign, int m_tiles, int E)
{
    // an upper bound on the number of items: chunks <= E + n_assign / NMAX
    const int64_t max_items = ((int64_t)E + n_assign / NMAX + 1) * m_tiles;
    return (int)(ctas < max_items ? ctas : max_items);
}

}  // namespace

template <int KIND>
cudaError_t set_smem()
{
    return cudaFuncSetAttribute(grouped_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<KIND>::SMEM);
}

cudaError_t gemm_init_device()
{
    cudaError_t e = set_smem<kGateUp>();
    if (e == cudaSuccess) e = set_smem<kDown>();
    if (e == cudaSuccess) e = set_smem<kGateUpRaw>();
    if (e == cudaSuccess) e = set_smem<kBwdQ>();
    if (e == cudaSuccess) e = set_smem<kBwdDx>();
    if (e == cudaSuccess) e = set_smem<kGateUpMx>();
    if (e == cudaSuccess) e = set_smem<kDownMx>();
    if (e == cudaSuccess) e = set_smem<kGateUpSave>();
    return e;
}

bool gemm_supported(int H, int I, int E)
{
    // TMA row coordinates are int32: the weight matrices' row counts must fit
    return H % 64 == 0 && I % 64 == 0 && (int64_t)E * 2 * I < INT32_MAX && (int64_t)E * H < INT32_MAX &&
           encoder() != nullptr;
}

namespace {

template <int KIND>
cudaError_t gate_up_like(const void *x, const int32_t *perm, int k, const void *wgu, const int4 *chunks,
                         const int32_t *nchunks, const int32_t *offs, int n_assign, int H, int I, int E, void *out0,
                         void *out1, int ctas, cudaStream_t s, float *g_keep = nullptr, float *u_keep = nullptr)
{
    CUtensorMap tA;
    constexpr int MT = Cfg<KIND>::MT;
    // groups of 16 neurons per box: MT tiles of 4, but never more than the tensor has
    const uint32_t groups = (uint32_t)(4 * MT < I / 16 ? 4 * MT : I / 16);
    cudaError_t e = make_gate_up_map(&tA, wgu, E, I, H, groups);
    if (e != cudaSuccess) return e;
    GemmArgs a{chunks, nchunks, offs, H, I, H, (I / 64 + MT - 1) / MT, I / 64, (int)groups * 32 * BK * 2, out0,
               out1, (const uint16_t *)x, perm, k};
    a.g_keep = g_keep;
    a.u_keep = u_keep;
    // the token rows come from x through the loader warps: the B maps are not read
    grouped_gemm_kernel<KIND><<<grid_for(ctas, n_assign, a.m_tiles, E), Cfg<KIND>::THREADS, Cfg<KIND>::SMEM, s>>>(
        tA, tA, tA, tA, tA, a);
    return cudaPeekAtLastError();
}

// The B maps of a hi/lo operand pair [rows][cols]: NMAX- and 16-row boxes.
cudaError_t make_pair_maps(CUtensorMap (&m)[4], const void *hi, const void *lo, uint64_t rows, uint64_t cols)
{
    cudaError_t e = make_map(&m[0], hi, rows, cols, SMALL_ROWS);
    if (e == cudaSuccess) e = make_map(&m[1], hi, rows, cols, NMAX);
    if (e == cudaSuccess) e = make_map(&m[2], lo, rows, cols, SMALL_ROWS);
    if (e == cudaSuccess) e = make_map(&m[3], lo, rows, cols, NMAX);
    return e;
}

// A 3-D BF16 map [d2][d1][d0] (d0 innermost) with a 64 x 64 x 1 box: 64
// elements of d0 (128 bytes, 128-byte swizzle) by 64 of d1.
cudaError_t make_mn_map(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {64, BK, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// q and dx: M (the weight side) of size m_size in tiles of 128, K = k_size.
template <int KIND>
cudaError_t launch_mn(const CUtensorMap &tA, const CUtensorMap (&tB)[4], const int4 *chunks, const int32_t *nchunks,
                      const int32_t *offs, int n_rows, int H, int I, int E, int m_size, int k_size, void *out0,
                      const BwdQArgs &q, int ctas, cudaStream_t s)
{
    constexpr int MT = Cfg<KIND>::MT;
    const int tiles = (m_size + BM - 1) / BM;
    GemmArgs a{chunks, nchunks, offs, H, I, k_size, (tiles + MT - 1) / MT, tiles, MT * BM * BK * 2, out0, nullptr,
               nullptr, nullptr, 0, q};
    grouped_gemm_kernel<KIND><<<grid_for(ctas, n_rows, a.m_tiles, E), Cfg<KIND>::THREADS, Cfg<KIND>::SMEM, s>>>(
        tA, tB[0], tB[1], tB[2], tB[3], a);
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t launch_gemm_gate_up(const void *x, const int32_t *perm, int k, const void *wgu, const int4 *chunks,
                                const int32_t *nchunks, const int32_t *offs, int n_assign, int H, int I, int E,
                                void *act_hi, void *act_lo, int ctas, cudaStream_t s)
{
    return gate_up_like<kGateUp>(x, perm, k, wgu, chunks, nchunks, offs, n_assign, H, I, E, act_hi, act_lo, ctas, s);
}

cudaError_t launch_gemm_gate_up_mx(const void *x, const int32_t *perm, int k, const void *gq, const void *gs,
                                   const int4 *chunks, const int32_t *nchunks, const int32_t *offs, int n_assign, int H,
                                   int I, int E, void *act_hi, void *act_lo, int ctas, cudaStream_t s)
{
    CUtensorMap tA;
    constexpr int MT = Cfg<kGateUpMx>::MT;
    const uint32_t groups = (uint32_t)(4 * MT < I / 16 ? 4 * MT : I / 16);
    cudaError_t e = make_gate_up_code_map(&tA, gq, E, I, H, groups);
    if (e != cudaSuccess) return e;
    GemmArgs a{chunks, nchunks, offs, H, I, H, (I / 64 + MT - 1) / MT, I / 64, (int)groups * 32 * BK, act_hi, act_lo,
               (const uint16_t *)x, perm, k, BwdQArgs{}, (const uint8_t *)gs, mx_scale_bytes(H)};
    grouped_gemm_kernel<kGateUpMx><<<grid_for(ctas, n_assign, a.m_tiles, E), Cfg<kGateUpMx>::THREADS,
                                     Cfg<kGateUpMx>::SMEM, s>>>(tA, tA, tA, tA, tA, a);
    return cudaPeekAtLastError();
}

cudaError_t launch_gemm_down_mx(const void *act_hi, const void *act_lo, const void *dq, const void *ds,
                                const int4 *chunks, const int32_t *nchunks, const int32_t *offs, int n_assign, int H,
                                int I, int E, float *z, int ctas, cudaStream_t s)
{
    CUtensorMap tA, tB[4];
    constexpr int MT = Cfg<kDownMx>::MT;
    cudaError_t e = make_down_code_map(&tA, dq, E, H, I);
    if (e == cudaSuccess) e = make_pair_maps(tB, act_hi, act_lo, n_assign, I);
    if (e != cudaSuccess) return e;
    const int tiles = (H + BM - 1) / BM;
    GemmArgs a{chunks, nchunks, offs, H, I, I, (tiles + MT - 1) / MT, tiles, MT * Cfg<kDownMx>::CODE_TILE, z, nullptr,
               nullptr, nullptr, 0, BwdQArgs{}, (const uint8_t *)ds, mx_scale_bytes(I)};
    grouped_gemm_kernel<kDownMx><<<grid_for(ctas, n_assign, a.m_tiles, E), Cfg<kDownMx>::THREADS,
                                   Cfg<kDownMx>::SMEM, s>>>(tA, tB[0], tB[1], tB[2], tB[3], a);
    return cudaPeekAtLastError();
}

cudaError_t launch_gemm_gate_up_raw(const void *x, const int32_t *perm, int k, const void *wgu, const int4 *chunks,
                                    const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E,
                                    float *g, float *u, int ctas, cudaStream_t s)
{
    return gate_up_like<kGateUpRaw>(x, perm, k, wgu, chunks, nchunks, offs, n_rows, H, I, E, g, u, ctas, s);
}

cudaError_t launch_gemm_gate_up_keep(const void *x, const int32_t *perm, int k, const void *wgu, const int4 *chunks,
                                     const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E,
                                     void *act_hi, void *act_lo, float *g, float *u, int ctas, cudaStream_t s)
{
    return gate_up_like<kGateUpSave>(x, perm, k, wgu, chunks, nchunks, offs, n_rows, H, I, E, act_hi, act_lo, ctas, s,
                                     g, u);
}

cudaError_t launch_bwd_q(const void *ds_hi, const void *ds_lo, const void *wd, const int4 *chunks,
                         const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E,
                         const BwdQOut &o, int ctas, cudaStream_t s)
{
    CUtensorMap tA, tB[4];
    cudaError_t e = make_mn_map(&tA, wd, I, H, E);
    if (e == cudaSuccess) e = make_pair_maps(tB, ds_hi, ds_lo, n_rows, H);
    if (e != cudaSuccess) return e;
    const BwdQArgs q{o.g, o.u, o.w_s, (__nv_bfloat16 *)o.dgu_hi, (__nv_bfloat16 *)o.dgu_lo,
                     (__nv_bfloat16 *)o.wa_hi, (__nv_bfloat16 *)o.wa_lo, o.dwp};
    return launch_mn<kBwdQ>(tA, tB, chunks, nchunks, offs, n_rows, H, I, E, I, H, nullptr, q, ctas, s);
}

cudaError_t launch_bwd_dx(const void *dgu_hi, const void *dgu_lo, const void *wgu, const int4 *chunks,
                          const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E, float *z,
                          int ctas, cudaStream_t s)
{
    CUtensorMap tA, tB[4];
    cudaError_t e = make_mn_map(&tA, wgu, H, 2 * (uint64_t)I, E);
    if (e == cudaSuccess) e = make_pair_maps(tB, dgu_hi, dgu_lo, n_rows, 2 * (uint64_t)I);
    if (e != cudaSuccess) return e;
    return launch_mn<kBwdDx>(tA, tB, chunks, nchunks, offs, n_rows, H, I, E, H, 2 * I, z, BwdQArgs{}, ctas, s);
}

cudaError_t launch_gemm_down(const void *act_hi, const void *act_lo, const void *wd, const int4 *chunks,
                             const int32_t *nchunks, const int32_t *offs, int n_assign, int H, int I, int E, float *z,
                             int ctas, cudaStream_t s)
{
    CUtensorMap tA, tB0s, tB0, tB1s, tB1;
    constexpr int MT = Cfg<kDown>::MT;
    cudaError_t e = make_down_map(&tA, wd, E, H, I);
    if (e == cudaSuccess) e = make_map(&tB0s, act_hi, n_assign, I, SMALL_ROWS);
    if (e == cudaSuccess) e = make_map(&tB0, act_hi, n_assign, I, NMAX);
    if (e == cudaSuccess) e = make_map(&tB1s, act_lo, n_assign, I, SMALL_ROWS);
    if (e == cudaSuccess) e = make_map(&tB1, act_lo, n_assign, I, NMAX);
    if (e != cudaSuccess) return e;
    const int tiles = (H + BM - 1) / BM;
    GemmArgs a{chunks, nchunks, offs, H, I, I, (tiles + MT - 1) / MT, tiles, MT * BM * BK * 2, z, nullptr, nullptr,
               nullptr, 0};
    grouped_gemm_kernel<kDown><<<grid_for(ctas, n_assign, a.m_tiles, E), kThreads, Cfg<kDown>::SMEM, s>>>(
        tA, tB0s, tB0, tB1s, tB1, a);
    return cudaPeekAtLastError();
}

}  // namespace moe
