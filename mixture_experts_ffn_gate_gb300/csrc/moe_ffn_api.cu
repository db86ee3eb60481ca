// moe_ffn_api.cu -- the C ABI: argument checks, workspace layout, path
// choice and the launch sequence of each path.  Host code only.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "moe_ffn.h"

namespace {

using moe::ceil_div;
using moe::round_up;

// Measured on GB300: the decode kernels win up to T = 4 (e.g. H4096 I1536
// E128 k8: 196 vs 237 us at T=4), the tensor-core grouped path from T = 8
// (H7168 I2048 E384 k8: 748 vs 979 us at T=8; 417 vs 697 us at H4096, T=16).
constexpr int kDefaultDecodeMaxTokens = 4;
constexpr int kDefaultWarps = 8;
// MXFP8 weights on the general decode kernels (CUDA cores): calls of up to
// kMxMaxTokens tokens when the caller forces the decode path.  AUTO takes
// them up to kMxDecodeTokens and the tensor-core grouped path beyond
// (measured on GB300: 2048-hidden layer T = 8 119 vs 134 us, 7168-hidden
// T = 8 735 vs 802 us; 4096-hidden T = 16 521 vs 408 us, T = 32 921 vs
// 508 us)
constexpr int kMxMaxTokens = 64;
constexpr int kMxDecodeTokens = 8;
constexpr int kMaxDevices = 64;

struct Shape {
    int64_t T, H, I, E, k;
};

// Workspace regions, 256-byte aligned.  First the fused decode kernel's
// state, which it keeps between calls: its flags (at offset 0 for every
// shape) and its tag region (right after them, its length depending on k
// and I), so calls of one k and I with any T share them and no other region
// of theirs overlaps them; a call of another shape may place its regions in
// a larger shape's tag region, which is why every call lowers the flags'
// size word to its own tag capacity (tag_cap).  Then the routing/sort
// region, shared by both paths; the rest is per path and the two overlap.
struct Layout {
    size_t flags, act_tag, idx, w, offs, perm, pos, uexp, ucount, chunks, nchunks, common_end;
    unsigned long long tag_cap;          // 64-bit words from act_tag to the next region
    size_t act;                          // decode: act f32 [T*k, I]
    size_t act_hi, act_lo, z;            // grouped
    size_t decode_total, grouped_total, total;
    // calls that pass the router weights: the logits [T, E] f32 (paths other
    // than the fused decode kernel) and the fused kernel's tagged logit words
    // (copies of [T*E] words of 16 bytes), after everything else
    size_t rlog, rtag, router_total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

Layout make_layout(const Shape &s)
{
    Layout L{};
    const size_t n = (size_t)(s.T * s.k);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    L.flags = take((size_t)moe::kDecodeFusedFlagWords * 8);
    L.act_tag = take(moe::decode_fused_tag_words((int)s.k, (int)s.I) * 8);
    L.idx = take(n * 4);
    L.tag_cap = (L.idx - L.act_tag) / 8;
    L.w = take(n * 4);
    L.offs = take((size_t)(s.E + 1) * 4);
    L.perm = take(n * 4);
    L.pos = take(n * 4);
    L.uexp = take((size_t)s.E * 4);
    L.ucount = take(4);
    L.chunks = take((size_t)(s.E + ceil_div((int64_t)n, moe::kGemmChunkMax) + 1) * 16);
    L.nchunks = take(4);
    L.common_end = o;
    // decode path: act f32 [T*k, I] (the general decode kernels, and the
    // fused decode kernel when it meets at its grid barrier)
    L.act = take(n * (size_t)s.I * 4);
    L.decode_total = o;
    // grouped path
    o = L.common_end;
    L.act_hi = take(n * (size_t)s.I * 2);
    L.act_lo = take(n * (size_t)s.I * 2);
    L.z = take(n * (size_t)s.H * 4);
    L.grouped_total = o;
    L.total = L.decode_total > L.grouped_total ? L.decode_total : L.grouped_total;
    o = L.total;
    L.rlog = take((size_t)(s.T * s.E) * 4);
    L.rtag = take((size_t)(s.T * s.E) * 16 * moe::kDecodeFusedLogitCopies);
    L.router_total = o;
    return L;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

int check_shape(const Shape &s)
{
    if (s.T < 0 || s.H < 1 || s.I < 1 || s.E < 1 || s.k < 1 || s.k > s.E) return MOE_ERR_INVALID_ARG;
    if (s.E > 1024 || s.k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (s.H % 64 || s.I % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (s.T * s.k > INT32_MAX / 2 || s.H > (1 << 24) || s.I > (1 << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

int check_args(const void *x, const float *logits, const void *wgu, const void *wd, const Shape &s,
               const float *out)
{
    int st = check_shape(s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;
    if (!x || !logits || !wgu || !wd || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(logits) || !aligned16(wgu) || !aligned16(wd) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

int check_opts(const moe_ffn_opts *o)
{
    if (!o) return MOE_OK;
    if (o->path < MOE_PATH_AUTO || o->path > MOE_PATH_GROUPED) return MOE_ERR_INVALID_ARG;
    if (o->decode_max_tokens < 0) return MOE_ERR_INVALID_ARG;
    if (o->gate_up_warps < 0 || o->gate_up_warps > 16) return MOE_ERR_INVALID_ARG;
    if (o->down_warps < 0 || o->down_warps > 16) return MOE_ERR_INVALID_ARG;
    if (o->gemm_ctas < 0) return MOE_ERR_INVALID_ARG;
    if (o->test_wait_limit_us < 0 || o->test_skip_arrival < 0) return MOE_ERR_INVALID_ARG;
    for (int r : o->reserved_in)
        if (r != 0) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Per-device set-up: kernel attributes and the SM count, done once per
// device and context (a new context, e.g. after cudaDeviceReset, has lost
// the kernel attributes).
struct DeviceInfo {
    bool ready = false;
    unsigned long long ctx = 0;
    int n_sm = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

int device_setup(DeviceInfo **info)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    const unsigned long long ctx = moe::current_context_id();
    if (!d.ready || d.ctx != ctx) {
        d.ready = false;
        if (cudaDeviceGetAttribute(&d.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::routing_init_device() != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::decode_init_device() != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::decode_fused_init_device() != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::gemm_init_device() != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::bwd_init_device() != cudaSuccess) return MOE_ERR_CUDA;
        // the attribute calls above created the context if there was none
        d.ctx = moe::current_context_id();
        d.ready = true;
    }
    *info = &d;
    return MOE_OK;
}

const char *kDecodeStages[] = {"router", "sort", "decode_gate_up", "decode_down"};
const char *kDecodeFusedStages[] = {"decode_fused"};
const char *kGroupedStages[] = {"router", "sort", "gemm_gate_up", "gemm_down", "combine"};
const char *kBackwardStages[] = {"router",  "sort",       "prep",       "gemm_gate_up",  "gemm_q", "gemm_dx",
                                 "combine", "zero_grads", "wgrad_down", "wgrad_gate_up", "dlogits"};
static_assert(sizeof kBackwardStages / sizeof *kBackwardStages <= MOE_MAX_STAGES, "stage events");
const char *kTrainForwardStages[] = {"router", "sort", "gemm_gate_up", "gemm_down", "combine"};
const char *kTrainBackwardStages[] = {"router",     "sort",       "prep",          "gemm_q",  "gemm_dx", "combine",
                                      "zero_grads", "wgrad_down", "wgrad_gate_up", "dlogits"};

// Records stage events around the launches of one call.  While the stream is
// being captured into a CUDA graph the records become external event-record
// nodes, so the events still time the graph's kernels when it is replayed.
struct Stages {
    cudaEvent_t *ev;
    cudaStream_t s;
    int n = 0;
    cudaError_t record(cudaEvent_t e)
    {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t r = cudaStreamIsCapturing(s, &cs);
        if (r != cudaSuccess) return r;
        return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                                                   : cudaEventRecord(e, s);
    }
    cudaError_t begin()
    {
        return ev ? record(ev[0]) : cudaSuccess;
    }
    cudaError_t done(cudaError_t launch)
    {
        if (launch != cudaSuccess) return launch;
        ++n;
        return ev ? record(ev[n]) : cudaSuccess;
    }
};

#define MOE_TRY(expr)                                \
    do {                                             \
        cudaError_t e_ = (expr);                     \
        if (e_ != cudaSuccess) return MOE_ERR_CUDA;  \
    } while (0)

// keep_state: the workspace is the caller's and keeps its contents between
// calls, so the fused decode kernel may use its tag region (a workspace
// allocated for one call is not: its memory may have held anything since).
// wr (nullable): the call passes the router weights [E, H] (and rbias [E],
// nullable) instead of logits; the logits are computed here (and copied to
// logits_out, nullable).  mx (nullable): MXFP8 expert weights instead of
// wgu/wd; such calls take the decode kernels only.  host_inputs: x and the
// logits are page-locked host memory read in place (not prefetched to L2).
int run_forward(const void *x, const float *logits, const void *wgu, const void *wd, const Shape &s, float *out,
                char *ws, const Layout &L, bool keep_state, int32_t *idx_out, float *w_out, moe_ffn_opts *opts,
                cudaStream_t stream, const void *wr = nullptr, const float *rbias = nullptr,
                float *logits_out = nullptr, const moe::FusedMx *mx = nullptr, bool host_inputs = false)
{
    DeviceInfo *dev = nullptr;
    int st = device_setup(&dev);
    if (st != MOE_OK) return st;

    const int T = (int)s.T, H = (int)s.H, I = (int)s.I, E = (int)s.E, k = (int)s.k;
    const int n_assign = T * k;
    int path = opts ? opts->path : MOE_PATH_AUTO;
    if (path == MOE_PATH_AUTO) {
        const int dlim = (opts && opts->decode_max_tokens) ? opts->decode_max_tokens
                         : mx                                ? kMxDecodeTokens
                                                             : kDefaultDecodeMaxTokens;
        path = (T <= dlim || !moe::gemm_supported(H, I, E)) ? MOE_PATH_DECODE : MOE_PATH_GROUPED;
    }
    if (path == MOE_PATH_GROUPED && !moe::gemm_supported(H, I, E)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int gu_warps = (opts && opts->gate_up_warps) ? opts->gate_up_warps : kDefaultWarps;
    const int dn_warps = (opts && opts->down_warps) ? opts->down_warps : kDefaultWarps;
    const int gemm_ctas = (opts && opts->gemm_ctas) ? opts->gemm_ctas : dev->n_sm;

    auto *idx = (int32_t *)(ws + L.idx);
    auto *w = (float *)(ws + L.w);
    auto *offs = (int32_t *)(ws + L.offs);
    auto *perm = (int32_t *)(ws + L.perm);
    auto *pos = (int32_t *)(ws + L.pos);
    auto *uexp = (int32_t *)(ws + L.uexp);
    auto *ucount = (int32_t *)(ws + L.ucount);
    auto *chunks = (int4 *)(ws + L.chunks);
    auto *nchunks = (int32_t *)(ws + L.nchunks);

    Stages stg{opts ? opts->stage_events : nullptr, stream};
    MOE_TRY(stg.begin());
    if (mx && path == MOE_PATH_DECODE && T > kMxMaxTokens) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (path == MOE_PATH_DECODE && (wr ? moe::decode_fused_router_supported(T, H, I, E, k, dev->n_sm)
                                       : moe::decode_fused_supported(T, H, I, E, k, dev->n_sm, mx != nullptr))) {
        // a few tokens: one cooperative kernel that routes them, streams both
        // projections' rows of the touched experts and exchanges the act
        // rows in between
        path = MOE_PATH_DECODE_FUSED;
        const unsigned long long wait_ns = (opts && opts->test_wait_limit_us)
                                               ? 1000ull * (unsigned long long)opts->test_wait_limit_us
                                               : moe::kDecodeFusedWaitNs;
        const moe::FusedRouter fr{wr, rbias, (unsigned long long *)(ws + L.rtag), logits_out};
        MOE_TRY(stg.done(moe::launch_decode_fused(
            x, logits, wgu, wd, T, H, I, E, k, dev->n_sm, (float *)(ws + L.act),
            keep_state ? (unsigned long long *)(ws + L.act_tag) : nullptr, L.tag_cap,
            (unsigned long long *)(ws + L.flags), idx_out, w_out, out, opts ? opts->exchange_out : nullptr, wait_ns,
            opts ? opts->test_skip_arrival : 0, wr ? &fr : nullptr, mx, !host_inputs, stream)));
        if (opts) {
            opts->n_stages = stg.n;
            opts->path_taken = path;
        }
        return MOE_OK;
    }
    // on a workspace that keeps state, the router also tells the fused
    // decode kernel's state which words this call's other regions overwrite
    auto *tag_size = keep_state ? (unsigned long long *)(ws + L.flags) + moe::kDecodeFusedSizeWord : nullptr;
    if (wr) {  // the router projection first; it and the top-k form the "router" stage
        logits = (const float *)(ws + L.rlog);
        MOE_TRY(moe::launch_router_gemv(x, wr, rbias, T, H, E, (float *)(ws + L.rlog), logits_out, stream));
    }
    MOE_TRY(stg.done(moe::launch_router(logits, T, E, k, idx, w, idx_out, w_out, tag_size, L.tag_cap, stream)));
    if (path == MOE_PATH_DECODE) {
        auto *act = (float *)(ws + L.act);
        MOE_TRY(stg.done(moe::launch_sort(idx, n_assign, E, moe::kGemmChunkMax, offs, perm, pos, uexp, ucount,
                                          nullptr, nullptr, stream)));
        MOE_TRY(stg.done(moe::launch_decode_gate_up(x, wgu, uexp, ucount, offs, perm, T, H, I, E, k, gu_warps,
                                                    act, mx, stream)));
        MOE_TRY(stg.done(moe::launch_decode_down(act, wd, w, uexp, ucount, offs, perm, T, H, I, k, dn_warps, out,
                                                 mx, stream)));
    } else {
        void *act_hi = ws + L.act_hi;
        void *act_lo = ws + L.act_lo;
        auto *z = (float *)(ws + L.z);
        MOE_TRY(stg.done(moe::launch_sort(idx, n_assign, E, moe::kGemmChunkMax, offs, perm, pos, uexp, ucount,
                                          chunks, nchunks, stream)));
        if (mx) {
            MOE_TRY(stg.done(moe::launch_gemm_gate_up_mx(x, perm, k, mx->gq, mx->gs, chunks, nchunks, offs, n_assign,
                                                         H, I, E, act_hi, act_lo, gemm_ctas, stream)));
            MOE_TRY(stg.done(moe::launch_gemm_down_mx(act_hi, act_lo, mx->dq, mx->ds, chunks, nchunks, offs,
                                                      n_assign, H, I, E, z, gemm_ctas, stream)));
        } else {
            MOE_TRY(stg.done(moe::launch_gemm_gate_up(x, perm, k, wgu, chunks, nchunks, offs, n_assign, H, I, E,
                                                      act_hi, act_lo, gemm_ctas, stream)));
            MOE_TRY(stg.done(moe::launch_gemm_down(act_hi, act_lo, wd, chunks, nchunks, offs, n_assign, H, I, E, z,
                                                   gemm_ctas, stream)));
        }
        MOE_TRY(stg.done(moe::launch_combine(z, w, pos, T, H, k, out, dev->n_sm, stream)));
    }
    if (opts) {
        opts->n_stages = stg.n;
        opts->path_taken = path;
    }
    return MOE_OK;
}

// ---------------------------------------------------------------- backward
// Workspace of moe_ffn_backward, 256-byte aligned regions.  The fused decode
// kernel's flags come first, where every forward layout has them, so a
// workspace shared with forward calls keeps their state consistent: this
// call's router lowers the state's size word to 0 (no tag region), and the
// next fused call re-prepares it.  Rows r index the padded sorted order:
// each expert's segment rounded up to 16 rows, at most 15 pad rows for each
// of the min(E, T*k) touched experts.
struct BwdLayout {
    size_t flags, idx, w, offs, perm, pos, uexp, ucount, chunks, nchunks, counts;
    size_t xs, ds_hi, ds_lo, w_s, g, u, dgu_hi, dgu_lo, wa_hi, wa_lo, dwp, z, total;
    int64_t rows;
};

BwdLayout make_bwd_layout(const Shape &s)
{
    BwdLayout L{};
    const int64_t n = s.T * s.k;
    L.rows = n + 15 * (s.E < n ? s.E : n);
    const size_t R = (size_t)L.rows;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    L.flags = take((size_t)moe::kDecodeFusedFlagWords * 8);
    L.idx = take((size_t)n * 4);
    L.w = take((size_t)n * 4);
    L.offs = take((size_t)(s.E + 1) * 4);
    L.perm = take(R * 4);
    L.pos = take((size_t)n * 4);
    L.uexp = take((size_t)s.E * 4);
    L.ucount = take(4);
    L.chunks = take((size_t)(s.E + ceil_div(L.rows, (int64_t)moe::kGemmChunkMax) + 1) * 16);
    L.nchunks = take(4);
    L.counts = take((size_t)s.E * 4);
    L.xs = take(R * (size_t)s.H * 2);
    L.ds_hi = take(R * (size_t)s.H * 2);
    L.ds_lo = take(R * (size_t)s.H * 2);
    L.w_s = take(R * 4);
    L.g = take(R * (size_t)s.I * 4);
    L.u = take(R * (size_t)s.I * 4);
    L.dgu_hi = take(R * (size_t)s.I * 4);
    L.dgu_lo = take(R * (size_t)s.I * 4);
    L.wa_hi = take(R * (size_t)s.I * 2);
    L.wa_lo = take(R * (size_t)s.I * 2);
    L.dwp = take(R * (size_t)(s.I / 32) * 4);
    L.z = take(R * (size_t)s.H * 4);
    L.total = o;
    return L;
}

// recompute: g and u recomputed from x (moe_ffn_backward); else they are in
// the workspace from moe_ffn_forward_train (moe_ffn_backward_train).  Both
// route and sort: everything that indexes memory is this call's own, so a
// state from another call can give wrong values but no stray access.
int run_backward(const void *x, const float *logits, const void *wgu, const void *wd, const float *dout,
                 const Shape &s, float *dx, float *dlogits, float *dwgu, float *dwd, char *ws, const BwdLayout &L,
                 moe_ffn_opts *opts, cudaStream_t stream, bool recompute = true)
{
    DeviceInfo *dev = nullptr;
    int st = device_setup(&dev);
    if (st != MOE_OK) return st;
    const int T = (int)s.T, H = (int)s.H, I = (int)s.I, E = (int)s.E, k = (int)s.k;
    const int rows = (int)L.rows;
    const int ctas = (opts && opts->gemm_ctas) ? opts->gemm_ctas : dev->n_sm;
    auto *idx = (int32_t *)(ws + L.idx);
    auto *w = (float *)(ws + L.w);
    auto *offs = (int32_t *)(ws + L.offs);
    auto *perm = (int32_t *)(ws + L.perm);
    auto *pos = (int32_t *)(ws + L.pos);
    auto *chunks = (int4 *)(ws + L.chunks);
    auto *nchunks = (int32_t *)(ws + L.nchunks);
    auto *counts = (int32_t *)(ws + L.counts);
    auto *g = (float *)(ws + L.g);
    auto *u = (float *)(ws + L.u);
    auto *w_s = (float *)(ws + L.w_s);
    auto *dwp = (float *)(ws + L.dwp);
    auto *z = (float *)(ws + L.z);
    auto *tag_size = (unsigned long long *)(ws + L.flags) + moe::kDecodeFusedSizeWord;

    Stages stg{opts ? opts->stage_events : nullptr, stream};
    MOE_TRY(stg.begin());
    MOE_TRY(stg.done(moe::launch_router(logits, T, E, k, idx, w, nullptr, nullptr, tag_size, 0, stream)));
    MOE_TRY(stg.done(moe::launch_sort(idx, T * k, E, moe::kGemmChunkMax, offs, perm, pos, (int32_t *)(ws + L.uexp),
                                      (int32_t *)(ws + L.ucount), chunks, nchunks, stream, 16, counts)));
    MOE_TRY(stg.done(moe::launch_bwd_prep(x, dout, w, perm, offs, rows, E, H, k, ws + L.xs, ws + L.ds_hi,
                                          ws + L.ds_lo, w_s, dev->n_sm, stream)));
    if (recompute)
        MOE_TRY(stg.done(moe::launch_gemm_gate_up_raw(x, perm, k, wgu, chunks, nchunks, offs, rows, H, I, E, g, u,
                                                      ctas, stream)));
    const moe::BwdQOut qo{g, u, w_s, ws + L.dgu_hi, ws + L.dgu_lo, ws + L.wa_hi, ws + L.wa_lo, dwp};
    MOE_TRY(stg.done(moe::launch_bwd_q(ws + L.ds_hi, ws + L.ds_lo, wd, chunks, nchunks, offs, rows, H, I, E, qo, ctas,
                                       stream)));
    MOE_TRY(stg.done(moe::launch_bwd_dx(ws + L.dgu_hi, ws + L.dgu_lo, wgu, chunks, nchunks, offs, rows, H, I, E, z,
                                        ctas, stream)));
    MOE_TRY(stg.done(moe::launch_combine(z, nullptr, pos, T, H, k, dx, dev->n_sm, stream)));
    MOE_TRY(stg.done(moe::launch_zero_untouched(counts, E, H, I, dwgu, dwd, dev->n_sm, stream)));
    MOE_TRY(stg.done(moe::launch_wgrad_down(ws + L.ds_hi, ws + L.ds_lo, ws + L.wa_hi, ws + L.wa_lo, offs, counts,
                                            rows, H, I, E, dwd, ctas, stream)));
    MOE_TRY(stg.done(moe::launch_wgrad_gate_up(ws + L.dgu_hi, ws + L.dgu_lo, ws + L.xs, offs, counts, rows, H, I, E,
                                               dwgu, ctas, stream)));
    MOE_TRY(stg.done(moe::launch_dlogits(dwp, pos, idx, w, T, E, k, I, dlogits, stream)));
    if (opts) {
        opts->n_stages = stg.n;
        opts->path_taken = recompute ? MOE_PATH_BACKWARD : MOE_PATH_TRAIN_BACKWARD;
    }
    return MOE_OK;
}

// The forward pass on the backward's workspace layout (the padded sorted
// order), keeping g and u in FP32 for the backward call, which routes and
// sorts the same logits again and finds them in the same rows.  act's hi/lo pair
// lives in the w*act regions, which the backward overwrites; the down GEMM's
// rows in z.  The kernels and their per-element order are the grouped
// forward's, so out has the same bits as a grouped moe_ffn_forward_ex call.
int run_forward_train(const void *x, const float *logits, const void *wgu, const void *wd, const Shape &s,
                      float *out, char *ws, const BwdLayout &L, moe_ffn_opts *opts, cudaStream_t stream)
{
    DeviceInfo *dev = nullptr;
    int st = device_setup(&dev);
    if (st != MOE_OK) return st;
    const int T = (int)s.T, H = (int)s.H, I = (int)s.I, E = (int)s.E, k = (int)s.k;
    const int rows = (int)L.rows;
    const int ctas = (opts && opts->gemm_ctas) ? opts->gemm_ctas : dev->n_sm;
    auto *idx = (int32_t *)(ws + L.idx);
    auto *w = (float *)(ws + L.w);
    auto *offs = (int32_t *)(ws + L.offs);
    auto *perm = (int32_t *)(ws + L.perm);
    auto *pos = (int32_t *)(ws + L.pos);
    auto *chunks = (int4 *)(ws + L.chunks);
    auto *nchunks = (int32_t *)(ws + L.nchunks);
    auto *counts = (int32_t *)(ws + L.counts);
    auto *z = (float *)(ws + L.z);
    auto *tag_size = (unsigned long long *)(ws + L.flags) + moe::kDecodeFusedSizeWord;

    Stages stg{opts ? opts->stage_events : nullptr, stream};
    MOE_TRY(stg.begin());
    MOE_TRY(stg.done(moe::launch_router(logits, T, E, k, idx, w, nullptr, nullptr, tag_size, 0, stream)));
    MOE_TRY(stg.done(moe::launch_sort(idx, T * k, E, moe::kGemmChunkMax, offs, perm, pos, (int32_t *)(ws + L.uexp),
                                      (int32_t *)(ws + L.ucount), chunks, nchunks, stream, 16, counts)));
    MOE_TRY(stg.done(moe::launch_gemm_gate_up_keep(x, perm, k, wgu, chunks, nchunks, offs, rows, H, I, E,
                                                   ws + L.wa_hi, ws + L.wa_lo, (float *)(ws + L.g),
                                                   (float *)(ws + L.u), ctas, stream)));
    MOE_TRY(stg.done(moe::launch_gemm_down(ws + L.wa_hi, ws + L.wa_lo, wd, chunks, nchunks, offs, rows, H, I, E, z,
                                           ctas, stream)));
    MOE_TRY(stg.done(moe::launch_combine(z, w, pos, T, H, k, out, dev->n_sm, stream)));
    if (opts) {
        opts->n_stages = stg.n;
        opts->path_taken = MOE_PATH_TRAIN_FORWARD;
    }
    return MOE_OK;
}

}  // namespace

namespace moe {

unsigned long long current_context_id()
{
    // the driver's cuCtxGetCurrent and cuCtxGetId, fetched through the
    // runtime (the library does not link libcuda); CUresult 0 is success
    using get_current_fn = int (*)(void **);
    using get_id_fn = int (*)(void *, unsigned long long *);
    static get_current_fn get_current = nullptr;
    static get_id_fn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) == cudaSuccess &&
            r1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) == cudaSuccess &&
            r2 == cudaDriverEntryPointSuccess) {
            get_current = (get_current_fn)p;
            get_id = (get_id_fn)q;
        }
        cudaGetLastError();
    });
    void *ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
    return id;
}

}  // namespace moe

static_assert(MOE_FFN_WORKSPACE_STATE_BYTES >= (size_t)moe::kDecodeFusedFlagWords * 8,
              "the state bytes must cover the fused decode kernel's flags");

extern "C" {

size_t moe_ffn_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k)
{
    Shape s{T, H, I, E, k};
    if (check_shape(s) != MOE_OK) return 0;
    return make_layout(s).total;
}

}  // extern "C"

namespace {

int forward_ex(const void *x_bf16, const float *router_logits_f32, const void *w_gate_up_bf16,
               const void *w_down_bf16, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, float *out_f32,
               void *workspace, size_t workspace_bytes, bool keep_state, int32_t *topk_idx_out, float *topk_w_out,
               moe_ffn_opts *opts, cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    int st = check_args(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, s, out_f32);
    if (st != MOE_OK) return st;
    st = check_opts(opts);
    if (st != MOE_OK) return st;
    if (opts) {
        opts->n_stages = 0;
        opts->path_taken = 0;
    }
    if (T == 0) return MOE_OK;
    if (!workspace || ((uintptr_t)workspace & 255)) return MOE_ERR_INVALID_ARG;
    if ((topk_idx_out && !aligned16(topk_idx_out)) || (topk_w_out && !aligned16(topk_w_out)))
        return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(s);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return run_forward(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, s, out_f32, (char *)workspace, L,
                       keep_state, topk_idx_out, topk_w_out, opts, stream);
}

}  // namespace

extern "C" {

int moe_ffn_forward_ex(const void *x_bf16, const float *router_logits_f32, const void *w_gate_up_bf16,
                       const void *w_down_bf16, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                       float *out_f32, void *workspace, size_t workspace_bytes, int32_t *topk_idx_out,
                       float *topk_w_out, moe_ffn_opts *opts, cudaStream_t stream)
{
    return forward_ex(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, T, H, I, E, k, out_f32, workspace,
                      workspace_bytes, true, topk_idx_out, topk_w_out, opts, stream);
}

size_t moe_ffn_router_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k)
{
    Shape s{T, H, I, E, k};
    if (check_shape(s) != MOE_OK) return 0;
    return make_layout(s).router_total;
}

int moe_ffn_forward_router(const void *x_bf16, const void *w_router_bf16, const float *router_bias_f32,
                           const void *w_gate_up_bf16, const void *w_down_bf16, int64_t T, int64_t H, int64_t I,
                           int64_t E, int64_t k, float *out_f32, void *workspace, size_t workspace_bytes,
                           float *logits_out, int32_t *topk_idx_out, float *topk_w_out, moe_ffn_opts *opts,
                           cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    int st = check_shape(s);
    if (st != MOE_OK) return st;
    st = check_opts(opts);
    if (st != MOE_OK) return st;
    if (opts) {
        opts->n_stages = 0;
        opts->path_taken = 0;
    }
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !w_router_bf16 || !w_gate_up_bf16 || !w_down_bf16 || !out_f32) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(w_router_bf16) || !aligned16(w_gate_up_bf16) || !aligned16(w_down_bf16) ||
        !aligned16(out_f32))
        return MOE_ERR_INVALID_ARG;
    if (router_bias_f32 && ((uintptr_t)router_bias_f32 & 3)) return MOE_ERR_INVALID_ARG;
    if ((logits_out && !aligned16(logits_out)) || (topk_idx_out && !aligned16(topk_idx_out)) ||
        (topk_w_out && !aligned16(topk_w_out)))
        return MOE_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255)) return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(s);
    if (workspace_bytes < L.router_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return run_forward(x_bf16, nullptr, w_gate_up_bf16, w_down_bf16, s, out_f32, (char *)workspace, L, true,
                       topk_idx_out, topk_w_out, opts, stream, w_router_bf16, router_bias_f32, logits_out);
}

int moe_ffn_forward_mxfp8(const void *x_bf16, const float *router_logits_f32, const void *w_gate_up_e4m3,
                          const void *w_gate_up_scale, const void *w_down_e4m3, const void *w_down_scale, int64_t T,
                          int64_t H, int64_t I, int64_t E, int64_t k, float *out_f32, void *workspace,
                          size_t workspace_bytes, int32_t *topk_idx_out, float *topk_w_out, moe_ffn_opts *opts,
                          cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    int st = check_shape(s);
    if (st != MOE_OK) return st;
    st = check_opts(opts);
    if (st != MOE_OK) return st;
    if (opts) {
        opts->n_stages = 0;
        opts->path_taken = 0;
    }
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !router_logits_f32 || !w_gate_up_e4m3 || !w_gate_up_scale || !w_down_e4m3 || !w_down_scale ||
        !out_f32)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(router_logits_f32) || !aligned16(w_gate_up_e4m3) ||
        !aligned16(w_gate_up_scale) || !aligned16(w_down_e4m3) || !aligned16(w_down_scale) || !aligned16(out_f32))
        return MOE_ERR_INVALID_ARG;
    if ((topk_idx_out && !aligned16(topk_idx_out)) || (topk_w_out && !aligned16(topk_w_out)))
        return MOE_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255)) return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(s);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const moe::FusedMx mx{w_gate_up_e4m3, w_gate_up_scale, w_down_e4m3, w_down_scale};
    return run_forward(x_bf16, router_logits_f32, nullptr, nullptr, s, out_f32, (char *)workspace, L, true,
                       topk_idx_out, topk_w_out, opts, stream, nullptr, nullptr, nullptr, &mx);
}

int moe_ffn_forward(const void *x_bf16, const float *router_logits_f32, const void *w_gate_up_bf16,
                    const void *w_down_bf16, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, float *out_f32,
                    cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    int st = check_args(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, s, out_f32);
    if (st != MOE_OK || T == 0) return st;
    const size_t bytes = make_layout(s).total;
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_NO_MEMORY;
    }
    st = forward_ex(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, T, H, I, E, k, out_f32, ws, bytes,
                    false, nullptr, nullptr, nullptr, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && st == MOE_OK) st = MOE_ERR_CUDA;
    return st;
}

size_t moe_ffn_host_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k)
{
    Shape s{T, H, I, E, k};
    if (check_shape(s) != MOE_OK) return 0;
    return align256((size_t)(T * H * 2)) + align256((size_t)(T * E * 4)) + align256((size_t)(T * H * 4)) +
           make_layout(s).total;
}

namespace {

// Inputs and output of at most this many bytes are read and written by the
// kernels in place when the host buffers are page-locked and mapped; larger
// ones are copied (the grouped path reads each token row k times).
constexpr size_t kDirectIoBytes = 1 << 20;

// The device address of page-locked, mapped host memory, or null.
const void *mapped_host(const void *p)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

int moe_ffn_forward_host(const void *x_host, const float *logits_host, const void *w_gate_up_bf16,
                         const void *w_down_bf16, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                         float *out_host, void *workspace, size_t workspace_bytes, moe_ffn_opts *opts,
                         cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    int st = check_shape(s);
    if (st != MOE_OK) return st;
    st = check_opts(opts);
    if (st != MOE_OK) return st;
    if (opts) {
        opts->n_stages = 0;
        opts->path_taken = 0;
    }
    if (T == 0) return MOE_OK;
    if (!x_host || !logits_host || !out_host || !w_gate_up_bf16 || !w_down_bf16) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_gate_up_bf16) || !aligned16(w_down_bf16)) return MOE_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < moe_ffn_host_workspace_bytes(T, H, I, E, k)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    char *p = (char *)workspace;
    const size_t xb = (size_t)(T * H * 2), lb = (size_t)(T * E * 4), ob = (size_t)(T * H * 4);
    if (xb + lb + ob <= kDirectIoBytes) {
        // small and page-locked: the kernels read x and the logits and write
        // out through the host link (NVLink-C2C on GB300), no copies
        const void *xd = mapped_host(x_host), *ld = mapped_host(logits_host), *od = mapped_host(out_host);
        if (xd && ld && od && aligned16(xd) && aligned16(ld) && aligned16(od)) {
            return run_forward(xd, (const float *)ld, w_gate_up_bf16, w_down_bf16, s, (float *)od, p,
                               make_layout(s), true, nullptr, nullptr, opts, stream, nullptr, nullptr, nullptr,
                               nullptr, true);
        }
    }
    // the device workspace first, so the fused decode kernel's state sits at
    // the same place for every T; then the staged inputs and output
    const Layout L = make_layout(s);
    char *ws = p;
    void *x_dev = p + L.total;
    auto *l_dev = (float *)(p + L.total + align256(xb));
    auto *o_dev = (float *)(p + L.total + align256(xb) + align256(lb));
    if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpyAsync(l_dev, logits_host, lb, cudaMemcpyHostToDevice, stream) != cudaSuccess) return MOE_ERR_CUDA;
    st = run_forward(x_dev, l_dev, w_gate_up_bf16, w_down_bf16, s, o_dev, ws, L, true, nullptr, nullptr, opts,
                     stream);
    if (st != MOE_OK) return st;
    if (cudaMemcpyAsync(out_host, o_dev, ob, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

size_t moe_ffn_backward_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k)
{
    Shape s{T, H, I, E, k};
    if (check_shape(s) != MOE_OK) return 0;
    return make_bwd_layout(s).total;
}

int moe_ffn_backward(const void *x_bf16, const float *router_logits_f32, const void *w_gate_up_bf16,
                     const void *w_down_bf16, const float *dout_f32, int64_t T, int64_t H, int64_t I, int64_t E,
                     int64_t k, float *dx_f32, float *dlogits_f32, float *dw_gate_up_f32, float *dw_down_f32,
                     void *workspace, size_t workspace_bytes, moe_ffn_opts *opts, cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    int st = check_shape(s);
    if (st != MOE_OK) return st;
    st = check_opts(opts);
    if (st != MOE_OK) return st;
    if (opts) {
        opts->n_stages = 0;
        opts->path_taken = 0;
        if (opts->path != MOE_PATH_AUTO && opts->path != MOE_PATH_GROUPED) return MOE_ERR_UNSUPPORTED_SHAPE;
    }
    if (!w_gate_up_bf16 || !w_down_bf16 || !dw_gate_up_f32 || !dw_down_f32) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_gate_up_bf16) || !aligned16(w_down_bf16) || !aligned16(dw_gate_up_f32) ||
        !aligned16(dw_down_f32))
        return MOE_ERR_INVALID_ARG;
    if (T > 0) {
        if (!x_bf16 || !router_logits_f32 || !dout_f32 || !dx_f32 || !dlogits_f32) return MOE_ERR_INVALID_ARG;
        if (!aligned16(x_bf16) || !aligned16(router_logits_f32) || !aligned16(dout_f32) || !aligned16(dx_f32) ||
            !aligned16(dlogits_f32))
            return MOE_ERR_INVALID_ARG;
    }
    const BwdLayout L = make_bwd_layout(s);
    if (L.rows > INT32_MAX / 2 || E * 2 * I * H >= ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (workspace && ((uintptr_t)workspace & 255)) return MOE_ERR_INVALID_ARG;
    if (workspace && T > 0 && workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    // the first check that asks the CUDA runtime (the TMA encoder)
    if (!moe::gemm_supported((int)H, (int)I, (int)E)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) {
        // no tokens: both weight gradients are zero
        if (cudaMemsetAsync(dw_gate_up_f32, 0, (size_t)(E * 2 * I * H) * 4, stream) != cudaSuccess ||
            cudaMemsetAsync(dw_down_f32, 0, (size_t)(E * H * I) * 4, stream) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (workspace)
        return run_backward(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, dout_f32, s, dx_f32, dlogits_f32,
                            dw_gate_up_f32, dw_down_f32, (char *)workspace, L, opts, stream);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, L.total, stream) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_NO_MEMORY;
    }
    st = run_backward(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, dout_f32, s, dx_f32, dlogits_f32,
                      dw_gate_up_f32, dw_down_f32, (char *)ws, L, opts, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && st == MOE_OK) st = MOE_ERR_CUDA;
    return st;
}

size_t moe_ffn_train_state_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k)
{
    return moe_ffn_backward_workspace_bytes(T, H, I, E, k);
}

namespace {

// The checks the training pair shares with moe_ffn_backward: shape, options,
// weights, the state buffer and its size.  None asks the CUDA runtime.
int check_train_call(const Shape &s, moe_ffn_opts *opts, const void *wgu, const void *wd, const void *state,
                     size_t state_bytes, BwdLayout *L)
{
    int st = check_shape(s);
    if (st != MOE_OK) return st;
    st = check_opts(opts);
    if (st != MOE_OK) return st;
    if (opts) {
        opts->n_stages = 0;
        opts->path_taken = 0;
        if (opts->path != MOE_PATH_AUTO && opts->path != MOE_PATH_GROUPED) return MOE_ERR_UNSUPPORTED_SHAPE;
    }
    if (!wgu || !wd || !state) return MOE_ERR_INVALID_ARG;
    if (!aligned16(wgu) || !aligned16(wd) || ((uintptr_t)state & 255)) return MOE_ERR_INVALID_ARG;
    *L = make_bwd_layout(s);
    if (L->rows > INT32_MAX / 2 || s.E * 2 * s.I * s.H >= ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (s.T > 0 && state_bytes < L->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return MOE_OK;
}

}  // namespace

int moe_ffn_forward_train(const void *x_bf16, const float *router_logits_f32, const void *w_gate_up_bf16,
                          const void *w_down_bf16, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                          float *out_f32, void *state, size_t state_bytes, moe_ffn_opts *opts, cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    BwdLayout L;
    int st = check_train_call(s, opts, w_gate_up_bf16, w_down_bf16, state, state_bytes, &L);
    if (st != MOE_OK) return st;
    if (T > 0) {
        if (!x_bf16 || !router_logits_f32 || !out_f32) return MOE_ERR_INVALID_ARG;
        if (!aligned16(x_bf16) || !aligned16(router_logits_f32) || !aligned16(out_f32)) return MOE_ERR_INVALID_ARG;
    }
    // the first check that asks the CUDA runtime (the TMA encoder)
    if (!moe::gemm_supported((int)H, (int)I, (int)E)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    return run_forward_train(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, s, out_f32, (char *)state, L,
                             opts, stream);
}

int moe_ffn_backward_train(const void *x_bf16, const float *router_logits_f32, const void *w_gate_up_bf16,
                           const void *w_down_bf16, const float *dout_f32, int64_t T, int64_t H, int64_t I,
                           int64_t E, int64_t k,
                           float *dx_f32, float *dlogits_f32, float *dw_gate_up_f32, float *dw_down_f32, void *state,
                           size_t state_bytes, moe_ffn_opts *opts, cudaStream_t stream)
{
    Shape s{T, H, I, E, k};
    BwdLayout L;
    int st = check_train_call(s, opts, w_gate_up_bf16, w_down_bf16, state, state_bytes, &L);
    if (st != MOE_OK) return st;
    if (!dw_gate_up_f32 || !dw_down_f32 || !aligned16(dw_gate_up_f32) || !aligned16(dw_down_f32))
        return MOE_ERR_INVALID_ARG;
    if (T > 0) {
        if (!x_bf16 || !router_logits_f32 || !dout_f32 || !dx_f32 || !dlogits_f32) return MOE_ERR_INVALID_ARG;
        if (!aligned16(x_bf16) || !aligned16(router_logits_f32) || !aligned16(dout_f32) || !aligned16(dx_f32) ||
            !aligned16(dlogits_f32))
            return MOE_ERR_INVALID_ARG;
    }
    // the first check that asks the CUDA runtime (the TMA encoder)
    if (!moe::gemm_supported((int)H, (int)I, (int)E)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) {
        if (cudaMemsetAsync(dw_gate_up_f32, 0, (size_t)(E * 2 * I * H) * 4, stream) != cudaSuccess ||
            cudaMemsetAsync(dw_down_f32, 0, (size_t)(E * H * I) * 4, stream) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    return run_backward(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, dout_f32, s, dx_f32, dlogits_f32,
                        dw_gate_up_f32, dw_down_f32, (char *)state, L, opts, stream, false);
}

const char *moe_ffn_status_string(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_NO_MEMORY: return "workspace allocation failed";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
    }
}

const char *moe_ffn_stage_name(int path, int stage)
{
    if (stage < 0) return nullptr;
    if (path == MOE_PATH_DECODE && stage < (int)(sizeof kDecodeStages / sizeof *kDecodeStages))
        return kDecodeStages[stage];
    if (path == MOE_PATH_DECODE_FUSED && stage < (int)(sizeof kDecodeFusedStages / sizeof *kDecodeFusedStages))
        return kDecodeFusedStages[stage];
    if (path == MOE_PATH_GROUPED && stage < (int)(sizeof kGroupedStages / sizeof *kGroupedStages))
        return kGroupedStages[stage];
    if (path == MOE_PATH_BACKWARD && stage < (int)(sizeof kBackwardStages / sizeof *kBackwardStages))
        return kBackwardStages[stage];
    if (path == MOE_PATH_TRAIN_FORWARD && stage < (int)(sizeof kTrainForwardStages / sizeof *kTrainForwardStages))
        return kTrainForwardStages[stage];
    if (path == MOE_PATH_TRAIN_BACKWARD && stage < (int)(sizeof kTrainBackwardStages / sizeof *kTrainBackwardStages))
        return kTrainBackwardStages[stage];
    return nullptr;
}

int moe_ffn_device_faults(uint32_t *flags, int clear)
{
    if (!flags) return MOE_ERR_INVALID_ARG;
    uint32_t gemm = 0, decode = 0, wgrad = 0;
    if (moe::read_fault_word(&gemm, clear != 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (moe::read_decode_fused_fault_word(&decode, clear != 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (moe::read_bwd_fault_word(&wgrad, clear != 0) != cudaSuccess) return MOE_ERR_CUDA;
    // bits 0-7: grouped GEMMs, 8-15: fused decode, 16-23: weight-gradient GEMMs
    *flags = gemm | (decode << 8) | (wgrad << 16);
    return MOE_OK;
}

}  // extern "C"
