// decode_fused.cu -- the decode path for a few tokens (T <= 4), as one kernel.
//
// The warp-decode article ("Cursor warp decode 공개 ...", section 핵심 내용)
// finishes a decode step in two kernels, one warp per output scalar, summing
// the routed experts' contributions in FP32 with no padding, scatter or
// per-expert buffers; its section 경쟁 구도 / 비교 keeps the intermediate
// activation unquantised.  On GB300 a decode step of up to four tokens is one
// cooperative launch, one CTA per SM, that moves the weights with bulk copies
// (cp.async.bulk) into a shared-memory ring:
//   - every CTA routes the tokens itself (the router kernel's warp top-k and
//     softmax, same bits) and lists the touched experts in ascending order,
//     each with its assignments a = t*k + j in ascending order, so every
//     touched expert's weights are streamed once;
//   - phase A: the CTA owns an equal, contiguous share of the U*I (expert u,
//     index i) pairs; pair (u, i) is gate row i and up row I+i of expert u.
//     For a run of pairs of one expert both row blocks are contiguous in
//     memory: the producer warp copies them into one ring slot (two bulk
//     copies), the consumer warps take the pairs round-robin, form both dot
//     products with every token the expert serves (x staged in shared memory
//     as BF16, widened to FP32 at use) and write
//     act = silu(gate) * up per assignment to global memory, in the two-plane
//     order phase B keeps in shared memory;
//   - the producer goes straight on to the CTA's W_down rows (dims
//     [h_lo, h_hi) of each touched expert, expert after expert, starting at
//     expert blockIdx.x % U when more than kRotateAbove are touched; they do
//     not depend on phase A), so they stream in while the act rows are
//     exchanged.  A ring slot takes as many of these rows as fit, across
//     expert boundaries (one bulk copy per expert run);
//   - phase B: once every act value is visible the CTA dots each of its
//     W_down rows with the act rows of the expert's assignments and finally
//     sums out[t, h] = sum_j w[t, j] * part[h][t*k + j] in slot order.  The
//     act rows are first copied into shared memory when all T*k of them fit
//     beside a ring of kMinSlots slots; otherwise they are read from global
//     memory as needed (one expert's rows at a time, so they stay in L1).
// Calls whose ring would still be shorter than kMinSlots use decode.cu.
// Each dot product uses decode.cu's lane split, chunk order, fmaf order and
// shuffle butterfly, so this path returns the same bits as the general decode
// path.  Every consumer warp visits every chunk in order (in phase B it reads
// the chunk's descriptor, written by the producer, and walks the chunk's
// expert runs only if one of its row groups lies there), so a ring slot's
// parity waits are never more than one phase ahead and the CTA-wide barriers
// match; every wait is bounded.
//
// Exchange of the act rows between phase A and phase B, in one of two ways.
// Every call has an epoch: a 64-bit salt drawn at random once per process
// plus twice a call counter kept in the workspace's flags array; every CTA
// reads the counter at its start and it is advanced once per call after all
// CTAs have read it, so no two calls on one flags array (eager or replayed
// from a CUDA graph) share an epoch within 2^31 calls.
//   - Grid barrier (two hops, every spin bounded): after a CTA-wide barrier
//     one thread of CTA b stores the low 32 bits of the epoch into arrival
//     word b (release).  In CTA 0, thread t watches words 4t..4t+3 with
//     16-byte relaxed loads until all hold the epoch, then issues an acq_rel
//     fence; after a CTA-wide barrier CTA 0 stores the epoch into the go word
//     (release), which one thread of every other CTA watches the same way,
//     and advances the counter.  Stale words never equal a later epoch, so
//     nothing needs zeroing.
//   - Tagged act (no barrier), for calls that stage the act rows in shared
//     memory: phase A writes each act value as one 64-bit word, epoch << 32
//     | float bits, into a tag region of the workspace, and phase B re-reads
//     the words (64-bit relaxed loads, single-copy atomic against the 64-bit
//     stores) until all carry the epoch: the data is its own flag, one hop
//     instead of the barrier's two plus the copy.  Every CTA stores the epoch
//     in its arrival word at its start; CTA 0's producer warp advances the
//     counter once all have.  A call trusts its T*k*I words of the tag
//     region only when the check word (a key xor the flags address) is set
//     and the size word is at least T*k*I.  The size word counts the leading
//     words of the region that hold nothing but zeros and tags of earlier
//     calls, which never equal the epoch (zero cannot: the epoch is odd):
//     a barrier call zeroes its T*k*I words before it raises the size word
//     to cover them, and every call on the workspace lowers the size word
//     to its tag_cap, the words of the region before the call's first other
//     region, because a call with a smaller k*I places its routing, act or
//     z rows inside the region of a larger one (this kernel does so
//     in CTA 0 once every CTA has read the flags; the other paths' router
//     kernel before anything else).  So memory that held other data never
//     stands in for an act value, whatever shapes share the workspace; only
//     the check word could match by chance (2^-64) in fresh memory.
#include <atomic>
#include <random>
#include <type_traits>


#include "common.cuh"
#include "kernels.h"
#include "route_block.cuh"
#include "sm100_ptx.cuh"

namespace moe {

__device__ uint32_t g_decode_fused_fault_word = 0;

// Opt-in timeline (build with -DMOE_FUSED_TIMELINE): each CTA records SM
// clock stamps of its phase boundaries and of every ring chunk's arrival as
// consumer warp 0 sees it, overwritten by every launch, read back with
// moe_ffn_debug_fused_timeline.  Slots per CTA (clock64 unless noted):
// 0 entry, 1 past griddepcontrol.wait, 2 routing done, 3 first copy issued,
// 4 last gate/up copy issued, 5 last W_down copy issued, 6 phase A done,
// 7 act exchange done, 8 act rows staged, 9 phase B done, 10 output
// written, 11 producer drained, 12 chunks seen, 13 phase A chunks, 14/15
// (calls with the router projection) its slices summed / every logit
// polled, 16..55 chunk c's full barrier passed, 56/57 token 0's routing
// warp before/after its selection, 58 flag words read, 62 globaltimer at
// the end, 63 globaltimer at entry.  The compiler may move a clock read across a block
// barrier, so stamps right after one are approximate.
#ifdef MOE_FUSED_TIMELINE
constexpr int kTimelineSlots = 64;
constexpr int kTimelineChunks = 40;
__device__ unsigned long long g_fused_timeline[kMaxGridCtas * kTimelineSlots];
#define MOE_TL(i) (g_fused_timeline[blockIdx.x * kTimelineSlots + (i)] = (unsigned long long)clock64())
#define MOE_TL_SET(i, v) (g_fused_timeline[blockIdx.x * kTimelineSlots + (i)] = (unsigned long long)(v))
#else
#define MOE_TL(i) ((void)0)
#define MOE_TL_SET(i, v) ((void)0)
#endif

namespace {

// Consumer warps per CTA.  With the producer warp that makes 16 warps, four
// per SM sub-partition, so each thread can hold 128 registers (a 17th warp
// would take a fifth slot on one sub-partition and cut that to 96).
constexpr int kConsumers = 15;
constexpr int kThreads = 32 * (1 + kConsumers);  // + the producer warp
constexpr int kChunkTarget = 32 * 1024;          // gate/up bytes per ring slot (whole row pairs)
constexpr int kChunkTargetOne = 16 * 1024;       // the same for one token, if it still holds two pairs
constexpr int kChunkTargetMx = 24 * 1024;        // the same for MXFP8 rows, if it holds two pairs
constexpr int kSlotMin = 16 * 1024;
constexpr int kMaxSlots = 16;
constexpr int kSmemCap = 224 * 1024;  // dynamic; the per-block limit also covers the static tables
constexpr int kMaxTokens = 4;
constexpr int kMaxAsg = 64;           // T * k
constexpr int kMinSlots = 5;          // ring slots the kernel needs (measured: 4 are too few)
// With more touched experts than this, each CTA starts its phase B rows at
// expert blockIdx.x % U instead of the first one (same results: the partial
// sums are combined in slot order).  Measured: the 2048- and 4096-hidden
// layers at four tokens (about 31 experts) run 4% and 7.6% faster, while at
// 8 and 16 experts the rotation gains nothing.
constexpr int kRotateAbove = 16;
// Tagged act words (16 bytes each) a consumer thread polls per batch, for up
// to two tokens and for more: under the weight stream an L2 round trip takes
// 1-2 us, so the fewer batches the better; 16 cover two tokens' 2 x 8 x 768
// act values of the 2048-hidden layer in one batch, and the four-token
// instance keeps 8 (16 would spill there).
constexpr int kPollWordsFew = 16, kPollWordsMany = 8;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr int kLogitReplicas = kDecodeFusedLogitCopies;  // copies of each published router logit

// flags (64-bit words): [0, kMaxGridCtas / 2) hold the kMaxGridCtas 32-bit
// arrival words, then the call counter, the tag-region check word and the
// tag-region size (64-bit words known to hold no live tag), then the go
// word on a 128-byte line of its own
constexpr int kCallWord = kMaxGridCtas;
constexpr int kCheckWord = kMaxGridCtas + 1;
constexpr int kSizeWord = kDecodeFusedSizeWord;
constexpr int kGoWord = kMaxGridCtas + 16;
static_assert(kGoWord < kDecodeFusedFlagWords, "flags array too small");
constexpr unsigned long long kCheckKey = 0x6d6f652d7461672dull;  // xor the flags address

// the kernel's mode bits: the test hook that skips the last CTA's arrival
// at the grid barrier, and the L2 prefetch of the inputs
constexpr int kSkipArrival = 1, kPrefetchInputs = 2;

// Named barriers of the one-token start (id 1 is the consumers' own):
// warp 0 publishes the ring's barriers and the flag words to the consumers
// (kBarPublish), the routing warp hands the touched experts to warp 0
// (kBarRouted), the consumers meet once the routing is in (kBarConsumers).
constexpr int kBarPublish = 2, kBarRouted = 3, kBarConsumers = 4;

enum : uint32_t {
    FAULT_LOGITS = 8u,
    FAULT_PRODUCER = 16u,
    FAULT_PHASE_A = 32u,
    FAULT_BARRIER = 64u,
    FAULT_PHASE_B = 128u,
};

// Shared-memory layout: ring | full[slots] | empty[slots] | flag | payload.
// The payload holds x [T][H] BF16 (phase A) and, in the same space, the act
// rows [T*k][I] FP32 of phase B if they are staged; then part [nh][T*k].
struct Layout {
    uint32_t full, empty, flag, payload, total;
};

__host__ __device__ inline Layout layout(int slots, int slot_bytes, uint32_t payload_bytes)
{
    Layout L;
    uint32_t o = (uint32_t)slots * slot_bytes;
    L.full = o;
    o += slots * 8;
    L.empty = o;
    o += slots * 8;
    L.flag = o;
    o += 16;
    L.payload = o;
    L.total = o + payload_bytes;
    return L;
}

__host__ __device__ inline uint32_t xa_bytes(int T, int H, int I, int k, bool act_in_smem)
{
    const uint32_t xb = (uint32_t)(2 * T * H), ab = act_in_smem ? (uint32_t)(4 * T * k * I) : 0u;
    return xb > ab ? xb : ab;
}

__device__ __forceinline__ void fail(volatile int *flag, uint32_t bit)
{
    if (!*flag) atomicOr(&g_decode_fused_fault_word, bit);
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

// Position in the ring of the next chunk: slot and the parity of the slot's
// current phase, advanced without divisions.
struct RingPos {
    int s = 0;
    uint32_t par = 0;
    __device__ __forceinline__ void next(int slots)
    {
        if (++s == slots) {
            s = 0;
            par ^= 1u;
        }
    }
};

// First task of consumer warp cw in a run whose first task has round-robin
// position `pos` (tasks go round-robin over the consumer warps).
__device__ __forceinline__ int first_task(int pos, int cw) { return (cw - pos + kConsumers) % kConsumers; }

// Position of element i of a row of n in the two-plane order: element 8u+e
// sits in plane e/4 at 4u + e%4.
__device__ __forceinline__ int plane_pos(int i, int n) { return ((i >> 2) & 1) * (n / 2) + (i >> 3) * 4 + (i & 3); }

// Spin (bounded, 16-byte relaxed loads) until the first n (<= 4) of the four
// words at p all hold v, then an acq_rel fence, which synchronises with the
// release stores that wrote them.
__device__ __forceinline__ bool wait_words4(const uint32_t *p, int n, uint32_t v, volatile int *flag,
                                            uint64_t t_start, uint64_t wait_ns)
{
    for (uint32_t spin = 0;; ++spin) {
        const uint4 w = ptx::ld_relaxed_gpu_v4(p);
        if (w.x == v && (n < 2 || w.y == v) && (n < 3 || w.z == v) && (n < 4 || w.w == v)) break;
        if ((spin & 63) == 63 && (*flag || ptx::globaltimer_ns() - t_start > wait_ns)) return false;
    }
    ptx::fence_acq_rel_gpu();
    return true;
}

// Gate and up dot products of one row pair (BF16 in shared memory) with the
// x rows of the expert's NB tokens (BF16 in shared memory, widened to FP32
// exactly); one lane
// per token writes act = silu(gate) * up of assignment asg[b] at column col
// of its global act row: as a plain float in act_g, or, when act_t is set, as
// one 64-bit word (tag << 32 | float bits) in act_t.  Each dot product keeps
// decode.cu's lane split, fmaf order and butterfly (split over the lanes,
// same pairs and bits).
template <int NB>
__device__ __forceinline__ void gate_up_pair(const uint8_t *grow, const uint8_t *urow, const uint16_t *const *xr,
                                             int H, int lane, const int *asg, float *act_g,
                                             unsigned long long *act_t, uint32_t tag, int I, int col)
{
    constexpr int N = pow2_ceil(2 * NB);  // gate of token b in slot b, up in slot NB + b
    float acc[N];
#pragma unroll
    for (int q = 0; q < N; ++q) acc[q] = 0.0f;
#pragma unroll 4
    for (int h = lane * 8; h < H; h += 256) {
        float gf[8], uf[8];
        unpack8(lds16(grow + 2 * h), gf);
        unpack8(lds16(urow + 2 * h), uf);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float xf[8];
            unpack8(lds16(xr[b] + h), xf);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                acc[b] = fmaf(gf[q], xf[q], acc[b]);
                acc[NB + b] = fmaf(uf[q], xf[q], acc[NB + b]);
            }
        }
    }
    // the butterfly's totals: for one token the plain butterfly (every lane
    // ends with gate and up), for more split over the lanes, where the first
    // lane of gate slot b fetches up slot NB + b from NB * 32 / N lanes up
    float t, u;
    int b;
    bool writer;
    if constexpr (NB == 1) {
        warp_sum_n(acc);
        t = acc[0];
        u = acc[1];
        b = 0;
        writer = lane == 0;
    } else {
        constexpr int W = 32 / N;
        t = warp_sum_split(acc, lane);
        u = __shfl_sync(0xffffffffu, t, (lane + NB * W) & 31);
        b = lane / W;
        writer = lane % W == 0 && b < NB;
    }
    if (writer) {
        const float a = swiglu(t, u);
        const size_t at = (size_t)asg[b] * I + col;
        if (act_t)
            ptx::st_relaxed_gpu(act_t + at, ((unsigned long long)tag << 32) | __float_as_uint(a));
        else
            act_g[at] = a;
    }
}

// Phase B rows per warp task when a row serves NB assignments: NB * rows <= 4.
__host__ __device__ constexpr int rows_for(int nb) { return nb >= 3 ? 1 : 4 / nb; }

// Dot products of up to RB W_down rows (rowp, BF16 in shared memory; rows
// past nu repeat a valid row and are dropped) with the act rows arow[b] of
// the expert's NB assignments (two-plane FP32 in shared memory).  One lane
// per (row r, assignment b) stores it to part[r * A + asg[b]].  Each dot
// product keeps decode.cu's lane split, fmaf order and butterfly (split over
// the lanes, same pairs and bits).
template <int NB>
__device__ __forceinline__ void down_rows(const uint8_t *const *rowp, const float *const *arow, int I, int lane,
                                          int nu, const int *asg, float *part, int A)
{
    constexpr int RB = rows_for(NB);
    constexpr int N = pow2_ceil(RB * NB);  // row r, assignment b in slot r * NB + b
    float acc[N];
#pragma unroll
    for (int q = 0; q < N; ++q) acc[q] = 0.0f;
#pragma unroll 2
    for (int i = lane * 8; i < I; i += 256) {
        float af[NB][8];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float4 v0 = *reinterpret_cast<const float4 *>(arow[b] + i / 2);
            const float4 v1 = *reinterpret_cast<const float4 *>(arow[b] + I / 2 + i / 2);
            af[b][0] = v0.x; af[b][1] = v0.y; af[b][2] = v0.z; af[b][3] = v0.w;
            af[b][4] = v1.x; af[b][5] = v1.y; af[b][6] = v1.z; af[b][7] = v1.w;
        }
        uint4 wv[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) wv[r] = lds16(rowp[r] + 2 * i);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float wf[8];
            unpack8(wv[r], wf);
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[r * NB + b] = fmaf(wf[q], af[b][q], acc[r * NB + b]);
        }
    }
    // the butterfly's totals, split over the lanes; the first lane of slot
    // r * NB + b stores it
    constexpr int W = 32 / N;
    const float t = warp_sum_split(acc, lane);
    const int slot = lane / W, r = slot / NB, b = slot - r * NB;
    if (lane % W == 0 && slot < RB * NB && r < nu) part[r * A + asg[b]] = t;
}

// ---- MXFP8 weights (the MX instantiation)
// E4M3 codes with one E8M0 scale per 32 elements along the reduction axis
// (the OCP MX specification's MXFP8).  The ring carries the codes and the
// scale bytes of the rows; each lane takes 16 consecutive elements per step
// (one 16-byte load), converts them to FP32 exactly (E4M3 -> F16 -> F32),
// forms its partial sums with the activations in FP32, and adds each partial
// sum times its block's scale (a power of two, so scaling the partial sum or
// every weight differ only in FP32 rounding order).

struct MxArgs {
    const uint8_t *gq, *gs;  // W_gate_up codes [E][2I][H] and scales [E][2I][hs]
    const uint8_t *dq, *ds;  // W_down codes [E][H][I] and scales [E][H][is]
    int hs, is;              // scale bytes per row (K / 32 padded to 16)
};

// gate_up_pair with MXFP8 rows: codes grow/urow, scale rows gsc/usc.
template <int NB>
__device__ __forceinline__ void gate_up_pair_mx(const uint8_t *grow, const uint8_t *urow, const uint8_t *gsc,
                                                const uint8_t *usc, const uint16_t *const *xr, int H, int lane,
                                                const int *asg, float *act_g, unsigned long long *act_t,
                                                uint32_t tag, int I, int col)
{
    constexpr int N = pow2_ceil(2 * NB);  // gate of token b in slot b, up in slot NB + b
    float acc[N];
#pragma unroll
    for (int q = 0; q < N; ++q) acc[q] = 0.0f;
#pragma unroll 2
    for (int h = lane * 16; h < H; h += 512) {
        float gf[16], uf[16];
        unpack16_e4m3(lds16(grow + h), gf);
        unpack16_e4m3(lds16(urow + h), uf);
        const float sg = e8m0_scale(gsc[h >> 5]), su = e8m0_scale(usc[h >> 5]);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float xf[16];
            unpack8(lds16(xr[b] + h), xf);
            unpack8(lds16(xr[b] + h + 8), xf + 8);
            float pg = 0.0f, pu = 0.0f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                pg = fmaf(gf[q], xf[q], pg);
                pu = fmaf(uf[q], xf[q], pu);
            }
            acc[b] = fmaf(pg, sg, acc[b]);
            acc[NB + b] = fmaf(pu, su, acc[NB + b]);
        }
    }
    float t, u;
    int b;
    bool writer;
    if constexpr (NB == 1) {
        warp_sum_n(acc);
        t = acc[0];
        u = acc[1];
        b = 0;
        writer = lane == 0;
    } else {
        constexpr int W = 32 / N;
        t = warp_sum_split(acc, lane);
        u = __shfl_sync(0xffffffffu, t, (lane + NB * W) & 31);
        b = lane / W;
        writer = lane % W == 0 && b < NB;
    }
    if (writer) {
        const float a = swiglu(t, u);
        const size_t at = (size_t)asg[b] * I + col;
        if (act_t)
            ptx::st_relaxed_gpu(act_t + at, ((unsigned long long)tag << 32) | __float_as_uint(a));
        else
            act_g[at] = a;
    }
}

// down_rows with MXFP8 rows: codes rowp[r], scale rows scp[r].  A lane
// takes LE = 16 consecutive elements per step, or 8 when I is not a
// multiple of 512 (then 16 would leave lanes idle in the last step: I = 768
// is one and a half steps of 16, three of 8).
template <int NB, int LE>
__device__ __forceinline__ void down_rows_mx(const uint8_t *const *rowp, const uint8_t *const *scp,
                                             const float *const *arow, int I, int lane, int nu, const int *asg,
                                             float *part, int A)
{
    static_assert(LE == 8 || LE == 16, "lane elements");
    constexpr int RB = rows_for(NB);
    constexpr int N = pow2_ceil(RB * NB);  // row r, assignment b in slot r * NB + b
    float acc[N];
#pragma unroll
    for (int q = 0; q < N; ++q) acc[q] = 0.0f;
    for (int i = lane * LE; i < I; i += 32 * LE) {
        // elements i .. i + LE - 1 of the two-plane act rows: LE / 8 groups
        // of 8 (group u: 4 values at 4u in plane 0, 4 at 4u in plane 1)
        float af[NB][LE];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
#pragma unroll
            for (int g = 0; g < LE / 8; ++g) {
                const float *p0 = arow[b] + i / 2 + 4 * g, *p1 = p0 + I / 2;
                const float4 v0 = *reinterpret_cast<const float4 *>(p0);
                const float4 v1 = *reinterpret_cast<const float4 *>(p1);
                af[b][8 * g + 0] = v0.x; af[b][8 * g + 1] = v0.y; af[b][8 * g + 2] = v0.z; af[b][8 * g + 3] = v0.w;
                af[b][8 * g + 4] = v1.x; af[b][8 * g + 5] = v1.y; af[b][8 * g + 6] = v1.z; af[b][8 * g + 7] = v1.w;
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float wf[16];
            if constexpr (LE == 16) {
                unpack16_e4m3(lds16(rowp[r] + i), wf);
            } else {
                const uint2 w2 = *reinterpret_cast<const uint2 *>(rowp[r] + i);
                unpack16_e4m3(make_uint4(w2.x, w2.y, 0u, 0u), wf);  // the first 8 values
            }
            const float sc = e8m0_scale(scp[r][i >> 5]);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float p = 0.0f;
#pragma unroll
                for (int q = 0; q < LE; ++q) p = fmaf(wf[q], af[b][q], p);
                acc[r * NB + b] = fmaf(p, sc, acc[r * NB + b]);
            }
        }
    }
    constexpr int W = 32 / N;
    const float t = warp_sum_split(acc, lane);
    const int slot = lane / W, r = slot / NB, b = slot - r * NB;
    if (lane % W == 0 && slot < RB * NB && r < nu) part[r * A + asg[b]] = t;
}

// down_rows_mx for a row group serving na (1 <= na <= NT) assignments.
template <int NT, int LE>
__device__ __forceinline__ void down_rows_mx_na(int na, const uint8_t *const *rowp, const uint8_t *const *scp,
                                                const float *const *arow, int I, int lane, int nu, const int *asg,
                                                float *part, int A)
{
    if (na == 1) down_rows_mx<1, LE>(rowp, scp, arow, I, lane, nu, asg, part, A);
    if constexpr (NT >= 2) {
        if (na == 2) down_rows_mx<2, LE>(rowp, scp, arow, I, lane, nu, asg, part, A);
    }
    if constexpr (NT >= 4) {
        if (na == 3) down_rows_mx<3, LE>(rowp, scp, arow, I, lane, nu, asg, part, A);
        if (na == 4) down_rows_mx<4, LE>(rowp, scp, arow, I, lane, nu, asg, part, A);
    }
}

// The router projection's inputs for the ROUTER instantiation: W_r [E][H]
// BF16, the bias [E] (nullable), the tagged logit words [T*E] (16 bytes
// each) and the caller's logits output (nullable).
struct RouterArgs {
    const uint16_t *wr;
    const float *bias;
    unsigned long long *ltag;
    float *logits_out;
    unsigned long long nonce;  // fresh for every launch from the host
};

// A 64-bit mixing function (the finaliser of Steele, Lea and Flood's
// SplitMix64): every input bit reaches every output bit.
__device__ __forceinline__ unsigned long long mix64(unsigned long long z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// ROUTER: the call passes the router weights instead of logits.  Before it
// routes, CTA b computes the logits o = b, b + grid, ... of the T*E -- the
// (logit, 256-element slice) pairs go round-robin over its warps
// (router_slice_warp), one thread per logit then adds the slices in order
// (router_logit_sum), the same arithmetic as the router kernel -- and
// publishes each as a 16-byte word:
// the call's 64-bit id, then the id's upper half << 32 | the logit's bits.
// The id mixes a nonce the host draws for every launch with the workspace's
// call counter, so no two calls of the process share one: replays of a
// captured launch keep its nonce but each advances the counter, while a
// workspace whose state was reset (counter back at zero, perhaps at the
// address of an earlier workspace) gets new nonces.  So a word left by any
// earlier call never matches, nor, but by chance (2^-96), other data; the
// words need no preparation.  Each half is single-copy atomic, so a reader
// that finds both halves carrying the id has the value of this call's store
// (a half from another store would carry another id's upper half, 2^-32).
// Every CTA polls all T*E words into its routing scratch and routes from
// there.  Each logit's word is stored in kLogitReplicas copies and CTA b
// polls copy b % kLogitReplicas, so the grid's polls spread over that many
// times more L2 lines (every CTA polls every logit, so one copy would draw
// all of them to the same few lines).
template <int NT, bool ROUTER, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fused_kernel(const uint16_t *__restrict__ x, const float *__restrict__ logits,
                        const uint16_t *__restrict__ wgu, const uint16_t *__restrict__ wd, int T, int H, int I, int E,
                        int k, int slots, int slot_bytes, int rpc, int rps, int nh_max, int act_in_smem,
                        float *__restrict__ act_g, unsigned long long *__restrict__ act_t,
                        unsigned long long tag_cap, unsigned long long *__restrict__ flags,
                        unsigned long long epoch_salt, int32_t *__restrict__ idx_out, float *__restrict__ w_out,
                        float *__restrict__ out, int32_t *__restrict__ exchange_out, uint64_t wait_ns,
                        int mode, RouterArgs ra, MxArgs mx)
{
    static_assert(!(ROUTER && MX), "the router projection is built for BF16 weights only");
    extern __shared__ __align__(128) uint8_t sm[];
    const int A = T * k;
    const uint32_t xa = xa_bytes(T, H, I, k, act_in_smem != 0);
    const Layout L = layout(slots, slot_bytes, xa + (uint32_t)nh_max * A * 4);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(sm + L.empty);
    volatile int *flag = reinterpret_cast<volatile int *>(sm + L.flag);
    // x as BF16 rows: a lane's 8 consecutive elements are one 16-byte load,
    // contiguous across the warp
    uint16_t *xs = reinterpret_cast<uint16_t *>(sm + L.payload);
    float *abuf = reinterpret_cast<float *>(sm + L.payload);  // phase B: act of all assignments [A][I]
    float *part = reinterpret_cast<float *>(sm + L.payload + xa);          // [nh][A]
    __shared__ int s_sel[kMaxAsg], s_asg[kMaxAsg], s_uexp[kMaxAsg], s_ubeg[kMaxAsg + 1], s_U;
    __shared__ int8_t s_rlog[kMaxAsg];  // per touched expert: log2 of the phase B rows per task
    __shared__ int s_xoff[kMaxAsg];     // per sorted assignment: its token's offset in xs
    __shared__ float s_w[kMaxAsg];
    __shared__ uint32_t s_key[kMaxAsg];
    // per ring slot, for its phase B chunk: first group id, number of
    // groups, expert and row of the chunk's first row (written by the
    // producer before it arms the slot's full barrier)
    __shared__ int4 s_desc[kMaxSlots];
    if (threadIdx.x == 0) {
        MOE_TL_SET(63, ptx::globaltimer_ns());
        MOE_TL(0);
    }
    // Launched with programmatic stream serialization: the next launch on
    // the stream may be scheduled from here on (its CTAs take an SM as one
    // of these exits), and nothing written by the previous launch -- the
    // caller's inputs included -- is read before it has completed.
    ptx::griddep_launch_dependents();
    // The tokens' logits and x rows, which every CTA reads first, fetched
    // into L2 while the previous launch drains (whole 16-byte pieces only)
    if ((mode & kPrefetchInputs) && threadIdx.x == 0 && blockIdx.x < 2) {
        const uint32_t n = blockIdx.x == 0 ? (ROUTER ? 0u : (uint32_t)(T * E * 4) & ~15u) : (uint32_t)(T * H * 2);
        if (n) ptx::bulk_prefetch_l2(blockIdx.x == 0 ? (const void *)logits : (const void *)x, n);
    }
    ptx::griddep_wait();
    if (threadIdx.x == 0) MOE_TL(1);
    if (threadIdx.x == 0) {
        for (int s = 0; s < slots; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, kConsumers);
        }
        *flag = 0;
        ptx::fence_barrier_init();
    }
    // this call's epoch and exchange mode come from words that no CTA
    // changes before every CTA has read them: thread 0 (not a routing warp)
    // reads them while the tokens are routed and shares them through shared
    // memory after the barrier that ends the routing
    const volatile unsigned long long *vflags = flags;
    __shared__ unsigned long long s_flags[3];  // call counter, check word, size word
    if (threadIdx.x == 0) {
        s_flags[0] = vflags[kCallWord];
        s_flags[1] = vflags[kCheckWord];
        s_flags[2] = vflags[kSizeWord];
#ifdef MOE_FUSED_TIMELINE
        if (s_flags[0] != ~0ull) MOE_TL(58);  // after the loads returned
#endif
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // One token (and logits passed in): its k experts are distinct, so the
    // routing warp lays out the touched list itself and the producer starts
    // its copies as soon as that warp is done, without waiting for the
    // block; the consumers meet on their own barriers.
    constexpr bool kFastStart = NT == 1 && !ROUTER;
    if constexpr (kFastStart) {
        if (warp == 0) {
            __syncwarp();
            ptx::named_arrive(kBarPublish, kThreads);
        }
    }

    if constexpr (ROUTER) {
        // x of all tokens into shared memory for phase A, while the
        // projection below reads x and W_r from global memory
        for (int v = threadIdx.x; v < T * H / 8; v += kThreads)
            reinterpret_cast<uint4 *>(xs)[v] = ld_nc16(x + (size_t)v * 8);
        const int TE = T * E;
        const int n_mine = TE > (int)blockIdx.x ? (TE - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        const int ns = router_slices(H);
        // slice sums [n_mine][ns] in the ring, after the routing scratch
        double *slice = reinterpret_cast<double *>(sm + (((size_t)TE * 4 + 15) & ~(size_t)15));
        for (int u = warp; u < n_mine * ns; u += kThreads / 32) {
            const int j = u / ns, sl = u - j * ns;
            const int o = blockIdx.x + j * gridDim.x, t = o / E, e = o - t * E;
            const double d = router_slice_warp(x + (size_t)t * H, ra.wr + (int64_t)e * H, H, sl, lane);
            if (lane == 0) slice[u] = d;
        }
        __syncthreads();  // slices summed, x staged; thread 0 has read the flag words
        if (threadIdx.x == 0) MOE_TL(14);
        const unsigned long long e64 = mix64(ra.nonce ^ (s_flags[0] * 0x9e3779b97f4a7c15ull));
        const unsigned long long tag_hi = e64 & 0xffffffff00000000ull;
        if (threadIdx.x < n_mine) {
            const int j = threadIdx.x, o = blockIdx.x + j * gridDim.x, e = o % E;
            const float v = router_logit_sum(slice + (size_t)j * ns, ns, ra.bias ? __ldg(ra.bias + e) : 0.0f);
            if (ra.logits_out) ra.logits_out[o] = v;
#pragma unroll
            for (int c = 0; c < kLogitReplicas; ++c)
                ptx::st_relaxed_gpu_v2u64(ra.ltag + 2 * ((size_t)c * TE + o), e64, tag_hi | __float_as_uint(v));
        }
        float *vals = reinterpret_cast<float *>(sm);  // the routing scratch: token t's logits at t * E
        const unsigned long long *copy = ra.ltag + 2 * (size_t)(blockIdx.x % kLogitReplicas) * TE;
        const uint64_t t_start = ptx::globaltimer_ns();
        for (int o = threadIdx.x; o < TE && !*flag; o += kThreads) {
            for (uint32_t spin = 0;; ++spin) {
                const ulonglong2 w = ptx::ld_relaxed_gpu_v2u64(copy + 2 * (size_t)o);
                if (w.x == e64 && (w.y >> 32) == (tag_hi >> 32)) {
                    vals[o] = __uint_as_float((uint32_t)w.y);
                    break;
                }
                if ((spin & 15) == 15 && (*flag || ptx::globaltimer_ns() - t_start > wait_ns)) {
                    fail(flag, FAULT_LOGITS);
                    break;
                }
            }
        }
        if (__syncthreads_or(*flag != 0)) return;  // no copy has been issued yet
        if (threadIdx.x == 0) MOE_TL(15);
    }

    // routing: consumer warp 1 + t routes token t (scratch: the ring)
    if (warp >= 1 && warp <= T) {
        const int t = warp - 1;
        int e;
        float wt;
        if (t == 0 && lane == 0) MOE_TL(56);
        route_token_warp<ROUTER>(logits + (int64_t)t * E, E, k, reinterpret_cast<float *>(sm) + (size_t)t * E, e,
                                 wt);
#ifdef MOE_FUSED_TIMELINE
        if (t == 0 && lane == 0 && wt != -1.0f) MOE_TL(57);
#endif
        if (lane < k) {
            s_sel[t * k + lane] = e;
            s_w[t * k + lane] = wt;
        }
        if constexpr (kFastStart) {
            if (lane < k) {
                if (blockIdx.x == 0) {
                    if (idx_out) idx_out[lane] = e;
                    if (w_out) w_out[lane] = wt;
                }
                s_uexp[lane] = e;
                s_ubeg[lane] = lane;
                s_asg[lane] = lane;
                s_xoff[lane] = 0;
                s_rlog[lane] = (int8_t)(rows_for(1) == 4 ? 2 : rows_for(1) == 2 ? 1 : 0);
            }
            if (lane == 0) {
                s_U = k;
                s_ubeg[k] = k;
            }
            __syncwarp();
            ptx::named_arrive(kBarRouted, 64);
        }
    }
    if constexpr (kFastStart) {
        if (warp == 0) {
            ptx::named_sync(kBarRouted, 64);
        } else {
            ptx::named_sync(kBarPublish, kThreads);
            ptx::named_sync(kBarConsumers, kThreads - 32);
        }
    } else {
    __syncthreads();
    if (threadIdx.x < A) {
        const int a = threadIdx.x;
        if (blockIdx.x == 0) {
            if (idx_out) idx_out[a] = s_sel[a];
            if (w_out) w_out[a] = s_w[a];
        }
        s_key[a] = ((uint32_t)s_sel[a] << 8) | (uint32_t)a;  // unique: (expert, assignment)
        if (T == 1) {  // one token: its k experts are distinct, slot order will do
            s_uexp[a] = s_sel[a];
            s_ubeg[a] = a;
            s_asg[a] = a;
            if (a == 0) {
                s_U = k;
                s_ubeg[k] = k;
            }
        }
    }
    __syncthreads();
    if (T > 1 && threadIdx.x < A) {  // rank sort of the keys
        const uint32_t key = s_key[threadIdx.x];
        int r = 0;
        for (int b = 0; b < A; ++b) r += s_key[b] < key;
        s_asg[r] = (int)key;
    }
    if (T > 1) __syncthreads();
    if (T > 1 && warp == 0) {  // touched experts, ascending; then keep only the assignment in s_asg
        int base = 0;
        for (int r0 = 0; r0 < A; r0 += 32) {
            const int r = r0 + lane;
            const uint32_t key = r < A ? (uint32_t)s_asg[r] : 0u;
            const bool nw = r < A && (r == 0 || (key >> 8) != ((uint32_t)s_asg[r - 1] >> 8));
            const uint32_t m = __ballot_sync(0xffffffffu, nw);
            if (nw) {
                const int u = base + __popc(m & ((1u << lane) - 1u));
                s_uexp[u] = (int)(key >> 8);
                s_ubeg[u] = r;
            }
            base += __popc(m);
        }
        __syncwarp();
        for (int r = lane; r < A; r += 32) s_asg[r] = s_asg[r] & 0xff;
        if (lane == 0) {
            s_U = base;
            s_ubeg[base] = A;
        }
    }
    if (T > 1) __syncthreads();
    if (threadIdx.x < s_U) {
        const int na = s_ubeg[threadIdx.x + 1] - s_ubeg[threadIdx.x];
        s_rlog[threadIdx.x] = (int8_t)(rows_for(na) == 4 ? 2 : rows_for(na) == 2 ? 1 : 0);
    }
    if (threadIdx.x < A) s_xoff[threadIdx.x] = s_asg[threadIdx.x] / k * H;
    __syncthreads();
    }
    const int U = s_U;
    if (threadIdx.x == 0) MOE_TL(2);

    const unsigned long long calls = s_flags[0];
    const uint32_t e32 = (uint32_t)(epoch_salt + 2 * calls);
    const bool tag_region = act_in_smem && act_t;  // this call may use, or prepare, the tag region
    const unsigned long long check_key = kCheckKey ^ (unsigned long long)flags;
    const bool skip_arrival = (mode & kSkipArrival) != 0;
    const bool tagged = tag_region && !skip_arrival && s_flags[1] == check_key &&
                        s_flags[2] >= (unsigned long long)(T * k) * I;
    uint32_t *arrive = reinterpret_cast<uint32_t *>(flags);
    if (tagged && threadIdx.x == 0) ptx::st_relaxed_gpu(arrive + blockIdx.x, e32);  // "read the counter"
    if (exchange_out && blockIdx.x == 0 && threadIdx.x == 0) *exchange_out = tagged ? 2 : 1;

    // Phase A: pairs [lo, hi) of the U*I, pair p = (expert p / I, index p % I),
    // in chunks of at most rpc pairs that never cross an expert.  Phase B:
    // output dims [h_lo, h_hi) of all U experts, the row sequence
    // s -> (expert (u_first + s / nh) % U, dim h_lo + s % nh), in chunks of
    // rps rows that may cross experts.  Producer and consumers walk both sequences with running
    // (expert, index) state.
    // 32-bit products: the host admits only T * k * I * grid < 2^32
    const uint32_t pairs = (uint32_t)(U * I);
    const int lo = (int)(pairs * blockIdx.x / gridDim.x);
    const int hi = (int)(pairs * (blockIdx.x + 1) / gridDim.x);
    const int h_lo = (int)((uint32_t)H * blockIdx.x / gridDim.x);
    const int h_hi = (int)((uint32_t)H * (blockIdx.x + 1) / gridDim.x);
    const int u_first = U > kRotateAbove ? (int)(blockIdx.x % U) : 0;  // expert of phase B's first row
    const int nh = h_hi - h_lo;
    const int nrow = U * nh;
    const int nb = (nrow + rps - 1) / rps;

    if (warp == 0) {
        int c = 0;
        if (lane == 0) {
            bool ok = true;
            RingPos rp;
            int u = lo / I, i0 = lo - u * I;
            for (int p = lo; p < hi && ok; ++c, rp.next(slots)) {
                const int n = min(rpc, min(I - i0, hi - p));
                const int s = rp.s;
                if (!ptx::mbar_wait_bounded(empty + s, rp.par ^ 1u, flag, wait_ns)) {
                    fail(flag, FAULT_PRODUCER);
                    ok = false;
                    break;
                }
                if constexpr (MX) {
                    // gate codes, up codes, gate scales, up scales
                    const uint32_t bytes = (uint32_t)n * H, sb = (uint32_t)n * mx.hs;
                    const int64_t r0 = (int64_t)s_uexp[u] * 2 * I + i0;  // first gate row
                    uint8_t *dst = sm + (size_t)s * slot_bytes;
                    ptx::mbar_arrive_expect_tx(full + s, 2 * bytes + 2 * sb);
                    ptx::bulk_load(dst, mx.gq + r0 * H, bytes, full + s);
                    ptx::bulk_load(dst + bytes, mx.gq + (r0 + I) * H, bytes, full + s);
                    ptx::bulk_load(dst + 2 * bytes, mx.gs + r0 * mx.hs, sb, full + s);
                    ptx::bulk_load(dst + 2 * bytes + sb, mx.gs + (r0 + I) * mx.hs, sb, full + s);
                } else {
                    const uint32_t bytes = (uint32_t)n * 2 * H;  // one block: gate or up rows
                    const uint16_t *gate = wgu + ((int64_t)s_uexp[u] * 2 * I + i0) * H;
                    ptx::mbar_arrive_expect_tx(full + s, 2 * bytes);
                    ptx::bulk_load(sm + (size_t)s * slot_bytes, gate, bytes, full + s);
                    ptx::bulk_load(sm + (size_t)s * slot_bytes + bytes, gate + (int64_t)I * H, bytes, full + s);
                }
                if (c == 0) MOE_TL(3);
                p += n;
                i0 += n;
                if (i0 == I) {
                    i0 = 0;
                    ++u;
                }
            }
            MOE_TL(4);
            MOE_TL_SET(13, c);
            int uu = u_first, rr = 0, gq = 0;  // next row to copy; groups before this chunk
            for (int q = 0; q < nb && ok; ++q, ++c, rp.next(slots)) {
                const int len_q = min(rps, nrow - q * rps);
                const int s = rp.s;
                if (!ptx::mbar_wait_bounded(empty + s, rp.par ^ 1u, flag, wait_ns)) {
                    fail(flag, FAULT_PRODUCER);
                    ok = false;
                    break;
                }
                int ngq = 0;  // groups of the chunk: each run's rows in groups of 1 << s_rlog
                for (int off = 0, u2 = uu, r2 = rr; off < len_q;) {
                    const int len = min(len_q - off, nh - r2), lg = s_rlog[u2];
                    ngq += (len + (1 << lg) - 1) >> lg;
                    off += len;
                    r2 += len;
                    if (r2 == nh) {
                        r2 = 0;
                        if (++u2 == U) u2 = 0;
                    }
                }
                s_desc[s] = make_int4(gq, ngq, uu, rr);
                gq += ngq;
                // the arrive releases the descriptor to the consumers that wait on the slot
                // MX: the slot holds rps code rows, then their scale rows
                ptx::mbar_arrive_expect_tx(full + s, (uint32_t)len_q * (MX ? I + mx.is : 2 * I));
                for (int off = 0; off < len_q;) {  // one copy per expert run (two for MX)
                    const int len = min(len_q - off, nh - rr);
                    const int64_t row = (int64_t)s_uexp[uu] * H + h_lo + rr;
                    if constexpr (MX) {
                        uint8_t *dst = sm + (size_t)s * slot_bytes;
                        ptx::bulk_load(dst + (size_t)off * I, mx.dq + row * I, (uint32_t)len * I, full + s);
                        ptx::bulk_load(dst + (size_t)rps * I + (size_t)off * mx.is, mx.ds + row * mx.is,
                                       (uint32_t)len * mx.is, full + s);
                    } else {
                        ptx::bulk_load(sm + (size_t)s * slot_bytes + (size_t)off * 2 * I, wd + row * I,
                                       (uint32_t)len * 2 * I, full + s);
                    }
                    off += len;
                    rr += len;
                    if (rr == nh) {
                        rr = 0;
                        if (++uu == U) uu = 0;
                    }
                }
            }
        }
        if (lane == 0) MOE_TL(5);
        __syncwarp();
        if (tagged && blockIdx.x == 0) {
            // no grid barrier in this call: advance the call counter once
            // every CTA has read it (its arrival word holds the epoch).  It
            // is advanced even after a failed wait, so that no later call
            // reuses this epoch.
            const uint64_t t_start = ptx::globaltimer_ns();
            for (int v = lane; 4 * v < (int)gridDim.x && !*flag; v += 32)
                if (!wait_words4(arrive + 4 * v, min(4, (int)gridDim.x - 4 * v), e32, flag, t_start, wait_ns))
                    fail(flag, FAULT_BARRIER);
            __syncwarp();
            if (lane == 0) {
                flags[kCallWord] = calls + 1;
                if (s_flags[2] > tag_cap) flags[kSizeWord] = tag_cap;
            }
        }
        if (lane == 0) {
            drain(full, slots, c);
            MOE_TL(11);
        }
        return;
    }

    const int ct = threadIdx.x - 32, n_ct = kConsumers * 32;
    const int cw = warp - 1;
    if constexpr (!ROUTER) {  // (the router projection staged x already)
        for (int v = ct; v < T * H / 8; v += n_ct)  // x of all tokens, 16 bytes at a time
            reinterpret_cast<uint4 *>(xs)[v] = ld_nc16(x + (size_t)v * 8);
        ptx::named_sync(1, n_ct);
    }

    // phase A: for each pair, gate and up dot products with every token of
    // the expert; act per assignment to global memory (tagged
    // words when this call exchanges act without a grid barrier)
    unsigned long long *const act_w = tagged ? act_t : nullptr;
    RingPos rp;
#ifdef MOE_FUSED_TIMELINE
    int pos_c = 0;  // chunks consumer warp 0 has seen
#endif
    {
        int u = lo / I, i0 = lo - u * I, pos = 0;
        for (int p = lo; p < hi; rp.next(slots)) {
            const int n = min(rpc, min(I - i0, hi - p));
            const int s = rp.s;
            if (!ptx::mbar_wait_bounded(full + s, rp.par, flag, wait_ns)) {
                fail(flag, FAULT_PHASE_A);
                break;
            }
#ifdef MOE_FUSED_TIMELINE
            if (ct == 0 && pos_c < kTimelineChunks) MOE_TL(16 + pos_c);
            ++pos_c;
#endif
            const uint8_t *chunk = sm + (size_t)s * slot_bytes;
            int m = first_task(pos, cw);
            if (m < n) {  // every warp walks every chunk: set up only with work
                const int a0 = s_ubeg[u], na = s_ubeg[u + 1] - a0;  // 1 <= na <= T <= NT
                const uint16_t *xr[NT];
#pragma unroll
                for (int b = 0; b < NT; ++b) xr[b] = xs + s_xoff[a0 + (b < na ? b : 0)];
                for (; m < n; m += kConsumers) {
                    const int col = plane_pos(i0 + m, I);
                    if constexpr (MX) {
                        const uint8_t *grow = chunk + (size_t)m * H;
                        const uint8_t *urow = grow + (size_t)n * H;
                        const uint8_t *gsc = chunk + (size_t)2 * n * H + (size_t)m * mx.hs;
                        const uint8_t *usc = gsc + (size_t)n * mx.hs;
                        if (na == 1)
                            gate_up_pair_mx<1>(grow, urow, gsc, usc, xr, H, lane, s_asg + a0, act_g, act_w, e32, I, col);
                        if constexpr (NT >= 2) {
                            if (na == 2)
                                gate_up_pair_mx<2>(grow, urow, gsc, usc, xr, H, lane, s_asg + a0, act_g, act_w, e32, I,
                                                   col);
                        }
                        if constexpr (NT >= 4) {
                            if (na == 3)
                                gate_up_pair_mx<3>(grow, urow, gsc, usc, xr, H, lane, s_asg + a0, act_g, act_w, e32, I,
                                                   col);
                            if (na == 4)
                                gate_up_pair_mx<4>(grow, urow, gsc, usc, xr, H, lane, s_asg + a0, act_g, act_w, e32, I,
                                                   col);
                        }
                    } else {
                        const uint8_t *grow = chunk + (size_t)m * 2 * H;
                        const uint8_t *urow = grow + (size_t)n * 2 * H;
                        if (na == 1) gate_up_pair<1>(grow, urow, xr, H, lane, s_asg + a0, act_g, act_w, e32, I, col);
                        if constexpr (NT >= 2) {
                            if (na == 2)
                                gate_up_pair<2>(grow, urow, xr, H, lane, s_asg + a0, act_g, act_w, e32, I, col);
                        }
                        if constexpr (NT >= 4) {
                            if (na == 3)
                                gate_up_pair<3>(grow, urow, xr, H, lane, s_asg + a0, act_g, act_w, e32, I, col);
                            if (na == 4)
                                gate_up_pair<4>(grow, urow, xr, H, lane, s_asg + a0, act_g, act_w, e32, I, col);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty + s);
            p += n;
            pos = (pos + n) % kConsumers;
            i0 += n;
            if (i0 == I) {
                i0 = 0;
                ++u;
            }
        }
    }

    // Exchange of the act rows.  Tagged: no grid barrier; phase B polls the
    // tagged words until every one carries this call's epoch.  Otherwise the
    // grid meets at the two-hop barrier, and a call that could use the tag
    // region first clears its share of it (zero never equals an epoch, which
    // is odd) so that CTA 0 can then mark the region as usable.
    const int nact = A * I;
    if (ct == 0) MOE_TL(6);
    if (!tagged && tag_region) {
        const int w_lo = (int)((int64_t)nact * blockIdx.x / gridDim.x);
        const int w_hi = (int)((int64_t)nact * (blockIdx.x + 1) / gridDim.x);
        for (int v = w_lo + ct; v < w_hi; v += n_ct) act_t[v] = 0ull;
    }
    ptx::named_sync(1, n_ct);
    if (!tagged) {  // grid barrier: every CTA's act values written and visible
        uint32_t *go = reinterpret_cast<uint32_t *>(flags + kGoWord);
        const uint64_t t_start = ptx::globaltimer_ns();
        // (the test hook: the last CTA does not arrive, so the waits run out)
        const bool arrives = !(skip_arrival && blockIdx.x == gridDim.x - 1);
        if (ct == 0 && !*flag && arrives) ptx::st_release_gpu(arrive + blockIdx.x, e32);
        if (blockIdx.x == 0) {
            for (int v = ct; 4 * v < (int)gridDim.x && !*flag; v += n_ct)
                if (!wait_words4(arrive + 4 * v, min(4, (int)gridDim.x - 4 * v), e32, flag, t_start, wait_ns))
                    fail(flag, FAULT_BARRIER);
            ptx::named_sync(1, n_ct);
            if (ct == 0 && !*flag) ptx::st_release_gpu(go, e32);
        } else if (ct == 0 && !*flag) {
            if (!wait_words4(go, 1, e32, flag, t_start, wait_ns)) fail(flag, FAULT_BARRIER);
        }
    }
    // every consumer leaves, or none: a producer fault can set the flag at any time
    const bool stop = ptx::named_sync_or(1, n_ct, *flag != 0);
    if (!tagged && blockIdx.x == 0 && ct == 0) {
        // past the barrier every CTA has read the flags and cleared its share
        // (or, after a failed wait, may still be clearing it: then the size
        // word is not raised).  The act rows of a call that reads them in
        // place lie past tag_cap, like every other region of this call.
        flags[kCallWord] = calls + 1;
        unsigned long long size = s_flags[1] == check_key ? s_flags[2] : 0ull;
        if (tag_region && !stop && size < (unsigned long long)nact) size = (unsigned long long)nact;
        flags[kSizeWord] = size < tag_cap ? size : tag_cap;
        if (tag_region && !stop) flags[kCheckWord] = check_key;
    }
    if (stop) return;
    if (ct == 0) MOE_TL(7);

    // phase B: W_down rows, chunk by chunk.  Within a run of one expert's
    // rows, groups of up to rows_for(na) consecutive rows share the act
    // loads; the groups go round-robin over the consumer warps, counted across
    // runs and chunks.  First every assignment's act row into shared memory.
    {
        if (tagged) {
            // each thread takes 16-byte words (two tagged values) kPollWords
            // at a time and re-reads the ones that do not yet carry the epoch
            constexpr int kPollWords = NT <= 2 ? kPollWordsFew : kPollWordsMany;
            const int nw = nact / 2;
            const uint64_t t_start = ptx::globaltimer_ns();
            for (int v0 = ct; v0 < nw; v0 += kPollWords * n_ct) {
                uint32_t need = 0;
#pragma unroll
                for (int j = 0; j < kPollWords; ++j)
                    if (v0 + j * n_ct < nw) need |= 1u << j;
                for (uint32_t spin = 0; need; ++spin) {
                    ulonglong2 w[kPollWords];
#pragma unroll
                    for (int j = 0; j < kPollWords; ++j)
                        if ((need >> j) & 1u) w[j] = ptx::ld_relaxed_gpu_v2u64(act_t + 2 * (size_t)(v0 + j * n_ct));
#pragma unroll
                    for (int j = 0; j < kPollWords; ++j)
                        if (((need >> j) & 1u) && (uint32_t)(w[j].x >> 32) == e32 && (uint32_t)(w[j].y >> 32) == e32) {
                            need &= ~(1u << j);
                            reinterpret_cast<float2 *>(abuf)[v0 + j * n_ct] =
                                make_float2(__uint_as_float((uint32_t)w[j].x), __uint_as_float((uint32_t)w[j].y));
                        }
                    if (need && (spin & 15) == 15 && (*flag || ptx::globaltimer_ns() - t_start > wait_ns)) {
                        fail(flag, FAULT_BARRIER);
                        break;
                    }
                }
                if (*flag) break;
            }
        } else if (act_in_smem) {
            const int n4 = nact / 4;
            for (int v0 = ct; v0 < n4; v0 += 4 * n_ct) {
                float4 a4[4];
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (v0 + b * n_ct < n4) a4[b] = __ldcg(reinterpret_cast<const float4 *>(act_g) + v0 + b * n_ct);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (v0 + b * n_ct < n4) reinterpret_cast<float4 *>(abuf)[v0 + b * n_ct] = a4[b];
            }
        }
        ptx::named_sync(1, n_ct);
        if (ct == 0) MOE_TL(8);
        // Two instances of the loop: with the act rows staged, their loads are
        // plain shared-memory loads (one pointer type for the compiler);
        // otherwise global loads through L1.
        auto rows_b = [&](auto staged) {
            const float *const act_base = decltype(staged)::value ? abuf : act_g;
            bool ok = true;
            for (int q = 0; q < nb; ++q, rp.next(slots)) {
                const int s = rp.s;
                if (ok && !ptx::mbar_wait_bounded(full + s, rp.par, flag, wait_ns)) {
                    fail(flag, FAULT_PHASE_B);
                    ok = false;
                }
#ifdef MOE_FUSED_TIMELINE
                if (ct == 0 && pos_c < kTimelineChunks) MOE_TL(16 + pos_c);
                ++pos_c;
#endif
                const int4 d = s_desc[s];
                // groups are numbered across runs and chunks; group g goes to warp
                // g % kConsumers.  A warp with none in this chunk skips its runs.
                int g = d.x + (cw - d.x % kConsumers + kConsumers) % kConsumers;
                if (ok && g < d.x + d.y) {
                    const uint8_t *chunk = sm + (size_t)s * slot_bytes;
                    const int len_q = min(rps, nrow - q * rps);
                    int uu = d.z, rr = d.w, gb = d.x;
                    for (int off = 0; off < len_q && g < d.x + d.y;) {
                        // rows [rr, rr + len) of expert uu: groups [gb, gb + ng)
                        const int len = min(len_q - off, nh - rr);
                        const int lg = s_rlog[uu];  // log2 of the rows per group
                        const int ng = (len + (1 << lg) - 1) >> lg;
                        if (g < gb + ng) {
                            const int a0 = s_ubeg[uu], na = s_ubeg[uu + 1] - a0;
                            const float *arow[NT];
#pragma unroll
                            for (int b = 0; b < NT; ++b)
                                arow[b] = act_base + (size_t)s_asg[a0 + (b < na ? b : 0)] * I;
                            float *pr = part + (size_t)rr * A;
                            for (; g < gb + ng; g += kConsumers) {
                                const int u0 = (g - gb) << lg, nu = min(1 << lg, len - u0);
                                const uint8_t *rowp[4];
                                float *const pu = pr + (size_t)u0 * A;
                                if constexpr (MX) {
                                    const uint8_t *scp[4];
#pragma unroll
                                    for (int r = 0; r < 4; ++r) {
                                        const size_t rw = (size_t)(off + u0 + (r < nu ? r : 0));
                                        rowp[r] = chunk + rw * I;
                                        scp[r] = chunk + (size_t)rps * I + rw * mx.is;
                                    }
                                    // 8-element lane steps unless I is a multiple of 512
                                    if (I % 512) {
                                        down_rows_mx_na<NT, 8>(na, rowp, scp, arow, I, lane, nu, s_asg + a0, pu, A);
                                    } else {
                                        down_rows_mx_na<NT, 16>(na, rowp, scp, arow, I, lane, nu, s_asg + a0, pu,
                                                                A);
                                    }
                                } else {
#pragma unroll
                                    for (int r = 0; r < 4; ++r)
                                        rowp[r] = chunk + (size_t)(off + u0 + (r < nu ? r : 0)) * 2 * I;
                                    if (na == 1) down_rows<1>(rowp, arow, I, lane, nu, s_asg + a0, pu, A);
                                    if constexpr (NT >= 2) {
                                        if (na == 2) down_rows<2>(rowp, arow, I, lane, nu, s_asg + a0, pu, A);
                                    }
                                    if constexpr (NT >= 4) {
                                        if (na == 3) down_rows<3>(rowp, arow, I, lane, nu, s_asg + a0, pu, A);
                                        if (na == 4) down_rows<4>(rowp, arow, I, lane, nu, s_asg + a0, pu, A);
                                    }
                                }
                            }
                        }
                        gb += ng;
                        off += len;
                        rr += len;
                        if (rr == nh) {
                            rr = 0;
                            if (++uu == U) uu = 0;
                        }
                    }
                }
                __syncwarp();
                if (ok && lane == 0) ptx::mbar_arrive(empty + s);
            }
        };
        if (act_in_smem)
            rows_b(std::true_type{});
        else
            rows_b(std::false_type{});
    }
    if (ct == 0) MOE_TL(9);
    if (ptx::named_sync_or(1, n_ct, *flag != 0)) return;
    for (int v = ct; v < T * nh; v += n_ct) {
        const int t = v / nh, r = v - t * nh;
        float o = 0.0f;
        for (int j = 0; j < k; ++j) o = fmaf(s_w[t * k + j], part[r * A + t * k + j], o);
        out[(size_t)t * H + h_lo + r] = o;
    }
#ifdef MOE_FUSED_TIMELINE
    if (ct == 0) {
        MOE_TL(10);
        MOE_TL_SET(12, pos_c);
        MOE_TL_SET(62, ptx::globaltimer_ns());
    }
#endif
}

// Geometry: phase A copies rpc whole gate/up row pairs (about kChunkTarget,
// or kChunkTargetOne, bytes); a slot holds the larger of that, kSlotMin and
// one W_down row, and phase B fills each slot with rps = slot / (bytes of a
// W_down row) rows.  As many slots as fit in shared memory beside the
// payload.  A BF16 row of K elements is 2K bytes; an MXFP8 row is K code
// bytes plus its scale row (mx_scale_bytes(K)).
struct Plan {
    int nt, rpc, rps, slot_bytes, slots, nh_max, act_in_smem;
    uint32_t payload;
};

Plan plan_for(int T, int H, int I, int k, int n_sm, bool mx = false)
{
    Plan p;
    p.nt = T <= 1 ? 1 : T <= 2 ? 2 : 4;
    p.nh_max = (H + n_sm - 1) / n_sm;
    const int pair_bytes = mx ? 2 * (H + mx_scale_bytes(H)) : 4 * H;
    const int row_bytes = mx ? I + mx_scale_bytes(I) : 2 * I;
    // one token does little work per byte: shorter chunks pipeline better
    // (measured: 2048-hidden layer 22.9 -> 22.1 us), as long as a chunk
    // keeps two pairs; with more tokens per pair, or one pair per chunk,
    // they are slower
    // MXFP8 chunks carry four copies (codes and scales of the gate and up
    // rows): 24 KB chunks while they hold two pairs (measured on the
    // 2048-hidden layer: T = 1 18.1 -> 17.1 us, T = 4 52.0 -> 49.9 us; one
    // pair per chunk made the 7168-hidden layer 15% slower)
    const int target = mx ? (kChunkTargetMx / pair_bytes >= 2 ? kChunkTargetMx : kChunkTarget)
                          : (T == 1 && kChunkTargetOne / pair_bytes >= 2) ? kChunkTargetOne : kChunkTarget;
    p.rpc = target / pair_bytes > 0 ? target / pair_bytes : 1;
    const int a = p.rpc * pair_bytes;
    int slot = a > kSlotMin ? a : kSlotMin;
    if (row_bytes > slot) slot = row_bytes;
    p.rps = slot / row_bytes;
    p.slot_bytes = slot;
    for (int staged = 1; staged >= 0; --staged) {  // act rows in shared memory if the ring keeps kMinSlots
        p.act_in_smem = staged;
        p.payload = xa_bytes(T, H, I, k, staged != 0) + (uint32_t)(p.nh_max * T * k * 4);
        const int fixed = (int)layout(0, p.slot_bytes, p.payload).total + 2 * kMaxSlots * 8;
        const int n = (kSmemCap - fixed) / p.slot_bytes;
        p.slots = n > kMaxSlots ? kMaxSlots : n;
        if (p.slots >= kMinSlots) break;
    }
    return p;
}

// A fresh 64-bit value for every launch that passes router weights: a
// process-wide counter started at a random point.
unsigned long long launch_nonce()
{
    static std::atomic<unsigned long long> next{[] {
        std::random_device rd;
        return ((unsigned long long)rd() << 32) ^ rd();
    }()};
    return next.fetch_add(1, std::memory_order_relaxed);
}

// The odd 64-bit salt of every epoch, drawn at random once per process.  A
// call's epoch is salt + 2 * (the flags array's call counter), so the calls
// on one flags array, eager or replayed from a CUDA graph, never repeat an
// epoch within 2^31 calls, and words left by another process or by other
// data match one only by chance (2^-32 per word).
unsigned long long epoch_salt()
{
    static const unsigned long long salt = [] {
        std::random_device rd;
        return (((unsigned long long)rd() << 32) ^ rd() ^ 0x9e3779b97f4a7c15ull) | 1ull;
    }();
    return salt;
}

}  // namespace

bool decode_fused_supported(int T, int H, int I, int E, int k, int n_sm, bool mx)
{
    if (T < 1 || T > kMaxTokens || T * k > kMaxAsg || n_sm > kMaxGridCtas) return false;
    // the kernel splits pairs and output dims over the CTAs in 32-bit arithmetic
    if ((uint64_t)T * k * I * n_sm >= (1ull << 32) || (uint64_t)H * n_sm >= (1ull << 32)) return false;
    if (mx && (H % 32 || I % 32)) return false;
    const Plan p = plan_for(T, H, I, k, n_sm, mx);
    return p.slots >= kMinSlots && (int64_t)T * E * 4 <= (int64_t)p.slots * p.slot_bytes;  // routing scratch
}

bool decode_fused_router_supported(int T, int H, int I, int E, int k, int n_sm)
{
    if (!decode_fused_supported(T, H, I, E, k, n_sm)) return false;
    // the routing scratch and the slice sums of the CTA's logits fit in the
    // ring; one thread per logit adds its slices
    const Plan p = plan_for(T, H, I, k, n_sm);
    const int64_t n_mine = ((int64_t)T * E + n_sm - 1) / n_sm;
    const int64_t need = (((int64_t)T * E * 4 + 15) & ~15) + n_mine * router_slices(H) * 8;
    return n_mine <= kThreads && need <= (int64_t)p.slots * p.slot_bytes;
}

size_t decode_fused_tag_words(int k, int I)
{
    const int a = kMaxTokens * k < kMaxAsg ? kMaxTokens * k : kMaxAsg;
    return (size_t)a * I;
}

cudaError_t launch_decode_fused(const void *x, const float *logits, const void *wgu, const void *wd, int T, int H,
                                int I, int E, int k, int n_sm, float *act, unsigned long long *act_tag,
                                unsigned long long tag_cap, unsigned long long *flags, int32_t *idx_out, float *w_out,
                                float *out, int32_t *exchange_out, unsigned long long wait_ns, int skip_arrival,
                                const FusedRouter *router, const FusedMx *mxw, bool prefetch_inputs,
                                cudaStream_t s)
{
    if (router && mxw) return cudaErrorInvalidValue;  // no such instantiation
    const Plan p = plan_for(T, H, I, k, n_sm, mxw != nullptr);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_sm);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = layout(p.slots, p.slot_bytes, p.payload).total;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // both act exchanges need every CTA resident
    attr[0].val.cooperative = 1;
    // the kernel waits for the previous launch before it reads anything, so
    // its CTAs may be scheduled while that launch drains (measured: 0.6 us
    // per call on the 2048-hidden layer in a CUDA graph)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    RouterArgs ra{};
    if (router)
        ra = RouterArgs{(const uint16_t *)router->wr, router->bias, router->ltag, router->logits_out, launch_nonce()};
    MxArgs ma{};
    if (mxw)
        ma = MxArgs{(const uint8_t *)mxw->gq, (const uint8_t *)mxw->gs, (const uint8_t *)mxw->dq,
                    (const uint8_t *)mxw->ds, mx_scale_bytes(H), mx_scale_bytes(I)};
    auto kern = router ? (p.nt == 1   ? decode_fused_kernel<1, true, false>
                          : p.nt == 2 ? decode_fused_kernel<2, true, false>
                                      : decode_fused_kernel<4, true, false>)
                : mxw  ? (p.nt == 1   ? decode_fused_kernel<1, false, true>
                          : p.nt == 2 ? decode_fused_kernel<2, false, true>
                                      : decode_fused_kernel<4, false, true>)
                       : (p.nt == 1   ? decode_fused_kernel<1, false, false>
                          : p.nt == 2 ? decode_fused_kernel<2, false, false>
                                      : decode_fused_kernel<4, false, false>);
    return cudaLaunchKernelEx(&cfg, kern, (const uint16_t *)x, logits, (const uint16_t *)wgu, (const uint16_t *)wd, T,
                              H, I, E, k, p.slots, p.slot_bytes, p.rpc, p.rps, p.nh_max, p.act_in_smem, act, act_tag,
                              tag_cap, flags, epoch_salt(), idx_out, w_out, out, exchange_out, (uint64_t)wait_ns,
                              (skip_arrival ? kSkipArrival : 0) | (prefetch_inputs ? kPrefetchInputs : 0), ra, ma);
}

cudaError_t read_decode_fused_fault_word(uint32_t *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_decode_fused_fault_word, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_decode_fused_fault_word, &zero, sizeof(uint32_t));
}

}  // namespace moe

#ifdef MOE_FUSED_TIMELINE
// Copies the timeline of the last fused decode launch (n_ctas x 64 words,
// layout above) to host memory; only in builds with -DMOE_FUSED_TIMELINE.
extern "C" int moe_ffn_debug_fused_timeline(unsigned long long *host, int n_ctas)
{
    if (!host || n_ctas < 1 || n_ctas > moe::kMaxGridCtas) return 1;
    return cudaMemcpyFromSymbol(host, moe::g_fused_timeline,
                                (size_t)n_ctas * moe::kTimelineSlots * sizeof(unsigned long long)) == cudaSuccess
               ? 0
               : 3;
}
#endif

namespace moe {

cudaError_t decode_fused_init_device()
{
    for (const void *kern :
         {(const void *)decode_fused_kernel<1, false, false>, (const void *)decode_fused_kernel<2, false, false>,
          (const void *)decode_fused_kernel<4, false, false>, (const void *)decode_fused_kernel<1, true, false>,
          (const void *)decode_fused_kernel<2, true, false>, (const void *)decode_fused_kernel<4, true, false>,
          (const void *)decode_fused_kernel<1, false, true>, (const void *)decode_fused_kernel<2, false, true>,
          (const void *)decode_fused_kernel<4, false, true>}) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace moe
