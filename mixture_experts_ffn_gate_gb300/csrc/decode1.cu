// decode1.cu -- the decode path for a single token (T = 1), as one kernel.
//
// The warp-decode article ("Cursor warp decode 공개 ...", section 핵심 내용)
// finishes a decode step in two kernels, one warp per output scalar, summing
// the routed experts' contributions in FP32 with no padding, scatter or
// per-expert buffers; its section 경쟁 구도 / 비교 keeps the intermediate
// activation unquantised.  On GB300 a single token's layer is one
// cooperative launch, one CTA per SM, that moves the weights with bulk
// copies (cp.async.bulk) into a shared-memory ring:
//   - every CTA routes the token itself (the router kernel's warp top-k and
//     softmax, same bits);
//   - phase A: the CTA owns an equal, contiguous share of the k*I (slot j,
//     index i) pairs; pair (j, i) is gate row i and up row I+i of expert
//     sel[j].  For a run of pairs of one slot both row blocks are contiguous
//     in memory: the producer warp copies them into one ring slot (two bulk
//     copies), the consumer warps take the pairs round-robin, form both dot
//     products with x (FP32) and write act = silu(gate) * up to global
//     memory, already in the two-plane order phase B keeps in shared memory;
//   - the producer goes straight on to the CTA's W_down rows (dims
//     [h_lo, h_hi) of each chosen expert, slot after slot; they do not
//     depend on phase A), so they stream in while the grid meets at a
//     barrier.  A ring slot takes as many of these rows as fit, across
//     expert boundaries (one bulk copy per expert run);
//   - phase B: after the barrier every CTA copies act (k*I FP32) into
//     shared memory, dots each of its W_down rows with act[j] and sums
//     out[h] = sum_j w_j * part[h][j] in slot order.
// Each dot product uses decode.cu's lane split, chunk order, fmaf order and
// shuffle butterfly, so this path returns the same bits as the general decode
// path.  Every consumer warp visits every chunk in order, so a ring slot's
// parity waits are never more than one phase ahead; every wait is bounded.
//
// Grid barrier (two hops, every spin bounded): after a CTA-wide barrier one
// thread of CTA b stores the low 32 bits of the call's epoch into arrival
// word b (release).  In CTA 0, thread t watches words 4t..4t+3 with 16-byte
// relaxed loads until all hold the epoch, then issues an acq_rel fence; after
// a CTA-wide barrier CTA 0 stores the epoch into the go word (release), which
// one thread of every other CTA watches the same way.  The epoch is the launch's odd 64-bit
// base (drawn at random per process, advanced per launch) plus twice a call
// counter kept in the flags array: every CTA reads the counter before it
// arrives and CTA 0 advances it after the barrier, so a CUDA-graph replay,
// which repeats the base, still gets a fresh epoch.  Stale words from earlier
// calls never equal a later epoch (within 2^31 calls), so nothing needs
// zeroing.
#include <atomic>
#include <random>

#include "common.cuh"
#include "kernels.h"
#include "route_block.cuh"
#include "sm100_ptx.cuh"

namespace moe {

__device__ uint32_t g_decode1_fault_word = 0;

namespace {

constexpr int kConsumers = 16;                   // consumer warps per CTA
constexpr int kThreads = 32 * (1 + kConsumers);  // + the producer warp
constexpr int kChunkTarget = 32 * 1024;          // gate/up bytes per ring slot (whole row pairs)
constexpr int kSlotMin = 16 * 1024;
constexpr int kRowsB = 4;                        // phase B rows per warp task
constexpr int kMaxSlots = 16;
constexpr int kSmemCap = 226 * 1024;  // dynamic; the per-block limit also covers static smem
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;

// flags (64-bit words): [0, kMaxGridCtas / 2) hold the kMaxGridCtas 32-bit
// arrival words, then the call counter, then the go word on a 128-byte line
// of its own
constexpr int kCallWord = kMaxGridCtas;
constexpr int kGoWord = kMaxGridCtas + 16;
static_assert(kGoWord < kDecode1FlagWords, "flags array too small");

enum : uint32_t {
    FAULT_PRODUCER = 16u,
    FAULT_PHASE_A = 32u,
    FAULT_BARRIER = 64u,
    FAULT_PHASE_B = 128u,
};

// Shared-memory layout: ring | full[slots] | empty[slots] | flag | vals[E] | payload
struct Layout {
    uint32_t full, empty, flag, vals, payload, total;
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
    L.vals = o;
    o += ((uint32_t)E * 4 + 15u) & ~15u;
    L.payload = o;
    L.total = o + payload_bytes;
    return L;
}

__host__ __device__ inline uint32_t xa_bytes(int H, int I, int k)
{
    return (uint32_t)(4 * H > 4 * k * I ? 4 * H : 4 * k * I);  // x in phase A, act in phase B
}

__device__ __forceinline__ void fail(volatile int *flag, uint32_t bit)
{
    if (!*flag) atomicOr(&g_decode1_fault_word, bit);
    *flag = 1;
}

__device__ __forceinline__ uint4 lds16(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

// The producer waits (bounded) until the last `slots` chunks it issued have
// landed, so no copy is in flight when the CTA exits.
__device__ __forceinline__ void drain(uint64_t *full, int slots, int issued)
{
    const volatile int keep = 0;
    for (int c = issued - 1; c >= 0 && c >= issued - slots; --c)
        ptx::mbar_wait_bounded(full + (c % slots), (uint32_t)(c / slots) & 1, &keep, kDrainNs);
}

// First task of consumer warp cw in a run whose first task has round-robin
// position `pos` (tasks go round-robin over the consumer warps).
__device__ __forceinline__ int first_task(int pos, int cw) { return (cw - pos + kConsumers) & (kConsumers - 1); }
static_assert((kConsumers & (kConsumers - 1)) == 0, "kConsumers must be a power of two");

// Position of act element i of a row in the two-plane order: element 8u+e
// sits in plane e/4 at 4u + e%4.
__device__ __forceinline__ int plane_pos(int i, int n) { return ((i >> 2) & 1) * (n / 2) + (i >> 3) * 4 + (i & 3); }


// Spin (bounded, 16-byte relaxed loads) until the first n (<= 4) of the four
// words at p all hold v, then an acq_rel fence, which synchronises with the
// release stores that wrote them.
__device__ __forceinline__ bool wait_words4(const uint32_t *p, int n, uint32_t v, volatile int *flag,
                                            uint64_t t_start)
{
    for (uint32_t spin = 0;; ++spin) {
        const uint4 w = ptx::ld_relaxed_gpu_v4(p);
        if (w.x == v && (n < 2 || w.y == v) && (n < 3 || w.z == v) && (n < 4 || w.w == v)) break;
        if ((spin & 63) == 63 && (*flag || ptx::globaltimer_ns() - t_start > kWaitNs)) return false;
    }
    ptx::fence_acq_rel_gpu();
    return true;
}

// Dot products of up to kRowsB W_down rows (rowp, BF16 in shared memory) with
// one act row (two-plane FP32 in shared memory); rows past nu repeat a valid
// row and are dropped.  Row r's result goes to part[r * k] (lane 0).  Each
// row keeps decode.cu's lane split, fmaf order and butterfly.
__device__ __forceinline__ void down_rows(const uint8_t *const (&rowp)[kRowsB], const float *arow, int I, int lane,
                                          int nu, float *part, int k)
{
    float acc[kRowsB];
#pragma unroll
    for (int r = 0; r < kRowsB; ++r) acc[r] = 0.0f;
#pragma unroll 2
    for (int i = lane * 8; i < I; i += 256) {
        const float4 v0 = *reinterpret_cast<const float4 *>(arow + i / 2);
        const float4 v1 = *reinterpret_cast<const float4 *>(arow + I / 2 + i / 2);
        const float af[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint4 wv[kRowsB];
#pragma unroll
        for (int r = 0; r < kRowsB; ++r) wv[r] = lds16(rowp[r] + 2 * i);
#pragma unroll
        for (int r = 0; r < kRowsB; ++r) {
            float wf[8];
            unpack8(wv[r], wf);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[r] = fmaf(wf[q], af[q], acc[r]);
        }
    }
    warp_sum_n(acc);
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRowsB; ++r)
            if (r < nu) part[r * k] = acc[r];
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode1_kernel(const uint16_t *__restrict__ x, const float *__restrict__ logits, const uint16_t *__restrict__ wgu,
                   const uint16_t *__restrict__ wd, int H, int I, int E, int k, int slots, int slot_bytes, int rpc,
                   int rps, int nh_max, float *__restrict__ act_g, unsigned long long *__restrict__ flags,
                   unsigned long long epoch_base, int32_t *__restrict__ idx_out, float *__restrict__ w_out,
                   float *__restrict__ out)
{
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t xa = xa_bytes(H, I, k);
    const Layout L = layout(slots, slot_bytes, E, xa + (uint32_t)nh_max * k * 4);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(sm + L.empty);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + L.flag);
    // x in FP32, two planes: element 8u+e sits in plane e/4 at 4u + e%4, so a
    // lane's 8 consecutive elements are two float4 loads that are contiguous
    // across the warp (no bank conflicts, no per-row unpacking).  Phase B
    // reuses the space for act [k][I], each row in the same two-plane form.
    float *xs = reinterpret_cast<float *>(sm + L.payload);
    float *act = xs;
    float *part = reinterpret_cast<float *>(sm + L.payload + xa);  // [nh][k]
    __shared__ int sel[32];
    __shared__ float wsm[32];
    if (threadIdx.x == 0) {
        for (int s = 0; s < slots; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, kConsumers);
        }
        *flag = 0;
        ptx::fence_barrier_init();
    }
    const unsigned long long calls = *reinterpret_cast<volatile unsigned long long *>(flags + kCallWord);
    const unsigned long long epoch = epoch_base + 2 * calls;
    route_token_block(logits, E, k, reinterpret_cast<float *>(sm + L.vals), sel, wsm);  // ends with __syncthreads
    if (blockIdx.x == 0 && threadIdx.x < k) {
        if (idx_out) idx_out[threadIdx.x] = sel[threadIdx.x];
        if (w_out) w_out[threadIdx.x] = wsm[threadIdx.x];
    }

    // Phase A: pairs [lo, hi) of the k*I, pair p = (slot p / I, index p % I),
    // in chunks of at most rpc pairs that never cross a slot.  Phase B:
    // output dims [h_lo, h_hi) of all k slots, the row sequence
    // s -> (slot s / nh, dim h_lo + s % nh), in chunks of rps rows that may
    // cross slots.  Producer and consumers walk both sequences with running
    // (slot, index) state.
    const int pairs = k * I;
    const int lo = (int)((int64_t)pairs * blockIdx.x / gridDim.x);
    const int hi = (int)((int64_t)pairs * (blockIdx.x + 1) / gridDim.x);
    const int h_lo = (int)((int64_t)H * blockIdx.x / gridDim.x);
    const int h_hi = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
    const int nh = h_hi - h_lo;
    const int nrow = k * nh;
    const int nb = (nrow + rps - 1) / rps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        if (lane == 0) {
            int c = 0;
            bool ok = true;
            int j = lo / I, i0 = lo - j * I;
            for (int p = lo; p < hi && ok; ++c) {
                const int n = min(rpc, min(I - i0, hi - p));
                const int s = c % slots;
                if (!ptx::mbar_wait_bounded(empty + s, ((uint32_t)(c / slots) & 1) ^ 1, flag, kWaitNs)) {
                    fail(flag, FAULT_PRODUCER);
                    ok = false;
                    break;
                }
                const uint32_t bytes = (uint32_t)n * 2 * H;  // one block: gate or up rows
                const uint16_t *gate = wgu + ((int64_t)sel[j] * 2 * I + i0) * H;
                ptx::mbar_arrive_expect_tx(full + s, 2 * bytes);
                ptx::bulk_load(sm + (size_t)s * slot_bytes, gate, bytes, full + s);
                ptx::bulk_load(sm + (size_t)s * slot_bytes + bytes, gate + (int64_t)I * H, bytes, full + s);
                p += n;
                i0 += n;
                if (i0 == I) {
                    i0 = 0;
                    ++j;
                }
            }
            int jj = 0, rr = 0;
            for (int q = 0; q < nb && ok; ++q, ++c) {
                const int len_q = min(rps, nrow - q * rps);
                const int s = c % slots;
                if (!ptx::mbar_wait_bounded(empty + s, ((uint32_t)(c / slots) & 1) ^ 1, flag, kWaitNs)) {
                    fail(flag, FAULT_PRODUCER);
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(full + s, (uint32_t)len_q * 2 * I);
                for (int off = 0; off < len_q;) {  // one copy per expert run
                    const int len = min(len_q - off, nh - rr);
                    ptx::bulk_load(sm + (size_t)s * slot_bytes + (size_t)off * 2 * I,
                                   wd + ((int64_t)sel[jj] * H + h_lo + rr) * I, (uint32_t)len * 2 * I, full + s);
                    off += len;
                    rr += len;
                    if (rr == nh) {
                        rr = 0;
                        ++jj;
                    }
                }
            }
            drain(full, slots, c);
        }
        return;
    }

    const int ct = threadIdx.x - 32, n_ct = kConsumers * 32;
    const int cw = warp - 1;
    for (int u = ct; u < H / 8; u += n_ct) {
        float f[8];
        unpack8(ld_nc16(x + (size_t)u * 8), f);
        *reinterpret_cast<float4 *>(xs + 4 * u) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4 *>(xs + H / 2 + 4 * u) = make_float4(f[4], f[5], f[6], f[7]);
    }
    ptx::named_sync(1, n_ct);

    // phase A: gate and up dot products of each pair, act to global memory
    int c = 0;
    {
        int j = lo / I, i0 = lo - j * I, pos = 0;
        for (int p = lo; p < hi; ++c) {
            const int n = min(rpc, min(I - i0, hi - p));
            const int s = c % slots;
            if (!ptx::mbar_wait_bounded(full + s, (uint32_t)(c / slots) & 1, flag, kWaitNs)) {
                fail(flag, FAULT_PHASE_A);
                break;
            }
            const uint8_t *chunk = sm + (size_t)s * slot_bytes;
            for (int m = first_task(pos, cw); m < n; m += kConsumers) {
                const uint8_t *grow = chunk + (size_t)m * 2 * H;
                const uint8_t *urow = grow + (size_t)n * 2 * H;
                float ag = 0.0f, au = 0.0f;
#pragma unroll 4
                for (int h = lane * 8; h < H; h += 256) {
                    float gf[8], uf[8];
                    unpack8(lds16(grow + 2 * h), gf);
                    unpack8(lds16(urow + 2 * h), uf);
                    const float4 x0 = *reinterpret_cast<const float4 *>(xs + h / 2);
                    const float4 x1 = *reinterpret_cast<const float4 *>(xs + H / 2 + h / 2);
                    const float xf[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        ag = fmaf(gf[q], xf[q], ag);
                        au = fmaf(uf[q], xf[q], au);
                    }
                }
                float gu2[2] = {ag, au};
                warp_sum_n(gu2);
                if (lane == 0) act_g[(size_t)j * I + plane_pos(i0 + m, I)] = swiglu(gu2[0], gu2[1]);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty + s);
            p += n;
            pos = (pos + n) & (kConsumers - 1);
            i0 += n;
            if (i0 == I) {
                i0 = 0;
                ++j;
            }
        }
    }

    // grid barrier: every CTA's act values written and visible
    ptx::named_sync(1, n_ct);
    {
        uint32_t *arrive = reinterpret_cast<uint32_t *>(flags);
        const uint32_t e32 = (uint32_t)epoch;
        const uint64_t t_start = ptx::globaltimer_ns();
        uint32_t *go = reinterpret_cast<uint32_t *>(flags + kGoWord);
        if (ct == 0 && !*flag) ptx::st_release_gpu(arrive + blockIdx.x, e32);
        if (blockIdx.x == 0) {
            for (int v = ct; 4 * v < (int)gridDim.x && !*flag; v += n_ct)
                if (!wait_words4(arrive + 4 * v, min(4, (int)gridDim.x - 4 * v), e32, flag, t_start))
                    fail(flag, FAULT_BARRIER);
            ptx::named_sync(1, n_ct);
            if (ct == 0 && !*flag) ptx::st_release_gpu(go, e32);
        } else if (ct == 0 && !*flag) {
            if (!wait_words4(go, 1, e32, flag, t_start)) fail(flag, FAULT_BARRIER);
        }
    }
    // every consumer leaves, or none: a producer fault can set the flag at any time
    const bool stop = ptx::named_sync_or(1, n_ct, *flag != 0);
    if (blockIdx.x == 0 && ct == 0) flags[kCallWord] = calls + 1;
    if (stop) return;

    // act of all k slots into shared memory (x's space), eight 16-byte loads
    // in flight per thread
    const int n4 = k * I / 4;
    for (int v0 = ct; v0 < n4; v0 += 8 * n_ct) {
        float4 a4[8];
#pragma unroll
        for (int b = 0; b < 8; ++b)
            if (v0 + b * n_ct < n4) a4[b] = __ldcg(reinterpret_cast<const float4 *>(act_g) + v0 + b * n_ct);
#pragma unroll
        for (int b = 0; b < 8; ++b)
            if (v0 + b * n_ct < n4) reinterpret_cast<float4 *>(act)[v0 + b * n_ct] = a4[b];
    }
    ptx::named_sync(1, n_ct);

    // phase B: W_down rows, chunk by chunk.  Within a run of one slot's rows,
    // groups of up to kRowsB consecutive rows share the act loads; the groups
    // go round-robin over the consumer warps, counted across runs and chunks.
    int jj = 0, rr = 0, pos = 0;
    for (int q = 0; q < nb; ++q, ++c) {
        const int len_q = min(rps, nrow - q * rps);
        const int s = c % slots;
        if (!ptx::mbar_wait_bounded(full + s, (uint32_t)(c / slots) & 1, flag, kWaitNs)) {
            fail(flag, FAULT_PHASE_B);
            break;
        }
        const uint8_t *chunk = sm + (size_t)s * slot_bytes;
        for (int off = 0; off < len_q;) {
            const int len = min(len_q - off, nh - rr);  // rows [rr, rr + len) of slot jj
            const int ng = (len + kRowsB - 1) / kRowsB;
            for (int g = first_task(pos, cw); g < ng; g += kConsumers) {
                const int u0 = g * kRowsB, nu = min(kRowsB, len - u0);
                const uint8_t *rowp[kRowsB];
#pragma unroll
                for (int r = 0; r < kRowsB; ++r)
                    rowp[r] = chunk + (size_t)(off + u0 + (r < nu ? r : 0)) * 2 * I;
                down_rows(rowp, act + (size_t)jj * I, I, lane, nu, part + (size_t)(rr + u0) * k + jj, k);
            }
            pos = (pos + ng) & (kConsumers - 1);
            off += len;
            rr += len;
            if (rr == nh) {
                rr = 0;
                ++jj;
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + s);
    }
    if (ptx::named_sync_or(1, n_ct, *flag != 0)) return;
    for (int r = ct; r < nh; r += n_ct) {
        float o = 0.0f;
        for (int j = 0; j < k; ++j) o = fmaf(wsm[j], part[r * k + j], o);
        out[h_lo + r] = o;
    }
}

// Geometry: phase A copies rpc whole gate/up row pairs (about kChunkTarget
// bytes); a slot holds the larger of that, kSlotMin and one W_down row, and
// phase B fills each slot with rps = slot / 2I rows.  As many slots as fit in
// shared memory beside the payload.
struct Plan {
    int rpc, rps, slot_bytes, slots, nh_max;
    uint32_t payload;
};

Plan plan_for(int H, int I, int E, int k, int n_sm)
{
    Plan p;
    p.nh_max = (H + n_sm - 1) / n_sm;
    p.rpc = kChunkTarget / (4 * H) > 0 ? kChunkTarget / (4 * H) : 1;
    const int a = p.rpc * 4 * H;
    int slot = a > kSlotMin ? a : kSlotMin;
    if (2 * I > slot) slot = 2 * I;
    p.rps = slot / (2 * I);
    p.slot_bytes = slot;
    p.payload = xa_bytes(H, I, k) + (uint32_t)(p.nh_max * k * 4);
    const int fixed = (int)layout(0, p.slot_bytes, E, p.payload).total + 2 * kMaxSlots * 8;
    const int n = (kSmemCap - fixed) / p.slot_bytes;
    p.slots = n > kMaxSlots ? kMaxSlots : n;
    return p;
}

std::atomic<unsigned long long> g_epoch{0};

// A value unique to this launch: a 64-bit counter whose start is drawn at
// random once per process, so flags left in a workspace by earlier calls (or
// by another process) do not match it.
unsigned long long next_epoch()
{
    static const unsigned long long base = [] {
        std::random_device rd;
        return ((unsigned long long)rd() << 32) ^ rd() ^ 0x9e3779b97f4a7c15ull;
    }();
    return base + 2 * g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
}

}  // namespace

bool decode1_supported(int H, int I, int E, int k, int n_sm)
{
    if (n_sm > kMaxGridCtas) return false;
    return plan_for(H, I, E, k, n_sm).slots >= 2;
}

cudaError_t launch_decode1(const void *x, const float *logits, const void *wgu, const void *wd, int H, int I, int E,
                           int k, int n_sm, float *act, unsigned long long *flags, int32_t *idx_out, float *w_out,
                           float *out, cudaStream_t s)
{
    const Plan p = plan_for(H, I, E, k, n_sm);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_sm);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = layout(p.slots, p.slot_bytes, E, p.payload).total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode1_kernel, (const uint16_t *)x, logits, (const uint16_t *)wgu,
                              (const uint16_t *)wd, H, I, E, k, p.slots, p.slot_bytes, p.rpc, p.rps, p.nh_max, act,
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
    return cudaFuncSetAttribute(decode1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
}

}  // namespace moe
