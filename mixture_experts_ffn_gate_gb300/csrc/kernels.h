// kernels.h -- launchers of the library's kernels (internal to libmoeffn.so).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Grouped path: at most this many assignments (token rows) per GEMM N-chunk.
constexpr int kGemmChunkMax = 64;

// MXFP8 expert weights of a call -- E4M3 codes gq [E, 2I, H] and dq [E, H,
// I], E8M0 scales gs [E, 2I, mx_scale_bytes(H)] and ds [E, H,
// mx_scale_bytes(I)] -- for the decode kernels (the weight pointers are then
// not read).
struct FusedMx {
    const void *gq, *gs, *dq, *ds;
};
// Bytes per scale row for rows of K elements: K / 32 scales padded to 16.
constexpr int mx_scale_bytes(int K) { return (K / 32 + 15) / 16 * 16; }

// routing.cu
cudaError_t routing_init_device();
// tag_size (nullable): the fused decode kernel's size word in a workspace
// that keeps its state; the router lowers it to tag_cap (the call's other
// regions start that many 64-bit words into the tag region).
cudaError_t launch_router(const float *logits, int T, int E, int k, int32_t *idx, float *w, int32_t *idx_copy,
                          float *w_copy, unsigned long long *tag_size, unsigned long long tag_cap, cudaStream_t s);
// logits [T, E] (and logits_copy, nullable) from x [T, H] and the router
// weights wr [E, H] (BF16) plus bias [E] (nullable): the exact sum rounded
// once to FP32
cudaError_t launch_router_gemv(const void *x, const void *wr, const float *bias, int T, int H, int E, float *logits,
                               float *logits_copy, cudaStream_t s);
size_t sort_smem_bytes(int E);
// pad > 1: every expert's segment rounded up to a multiple of pad rows (pad
// rows' perm = -1); counts (nullable): assignments per expert
cudaError_t launch_sort(const int32_t *idx, int n_assign, int E, int chunk_max, int32_t *offs, int32_t *perm,
                        int32_t *pos, int32_t *uexp, int32_t *ucount, int4 *chunks, int32_t *nchunks,
                        cudaStream_t s, int pad = 1, int32_t *counts = nullptr);
// w (nullable): without it the rows are summed unweighted
cudaError_t launch_combine(const float *z, const float *w, const int32_t *pos, int T, int H, int k, float *out,
                           int n_sm, cudaStream_t s);

// decode.cu
cudaError_t decode_init_device();
int decode_down_tok_tile(int T, int k);
cudaError_t launch_decode_gate_up(const void *x, const void *wgu, const int32_t *uexp, const int32_t *ucount,
                                  const int32_t *offs, const int32_t *perm, int T, int H, int I, int E, int k,
                                  int warps, float *act, const FusedMx *mxw, cudaStream_t s);
cudaError_t launch_decode_down(const float *act, const void *wd, const float *w, const int32_t *uexp,
                               const int32_t *ucount, const int32_t *offs, const int32_t *perm, int T, int H,
                               int I, int k, int warps, float *out, const FusedMx *mxw, cudaStream_t s);

// decode_fused.cu: a decode step of up to four tokens in one cooperative
// kernel.  act: [T*k][I] FP32 scratch; flags: kDecodeFusedFlagWords 64-bit
// words and act_tag: the tag region, both kept between calls (any initial
// contents); act_tag may be null (every call then meets at a grid barrier).
// Word kDecodeFusedSizeWord of flags counts the leading words of the tag
// region known to hold only zeros and tags.  Every call on a workspace that
// keeps state lowers it to its tag_cap, the 64-bit words of the tag region
// before the call's first other region: the fused kernel itself, and the
// router kernel on the other paths.
constexpr int kMaxGridCtas = 1024;
constexpr int kDecodeFusedFlagWords = kMaxGridCtas + 32;
constexpr int kDecodeFusedSizeWord = kMaxGridCtas + 2;
cudaError_t decode_fused_init_device();
cudaError_t read_decode_fused_fault_word(uint32_t *flags, bool clear);
// mx: with MXFP8 expert weights (FusedMx) instead of BF16 ones
bool decode_fused_supported(int T, int H, int I, int E, int k, int n_sm, bool mx = false);
// the same for a call that passes the router weights (its projection's
// scratch must fit too)
bool decode_fused_router_supported(int T, int H, int I, int E, int k, int n_sm);
size_t decode_fused_tag_words(int k, int I);
// exchange_out (nullable, device): CTA 0 stores 1 when the call met at the
// grid barrier, 2 when it exchanged tagged act words.  wait_ns bounds every
// wait; skip_arrival (a test hook) makes the last CTA skip its arrival at
// the grid barrier, so the call's waits run out and it reports a fault.
// router (nullable): the call passes the router weights instead of logits;
// the kernel computes the logits itself, exchanges them through ltag
// (kDecodeFusedLogitCopies copies of T*E words of 16 bytes, any initial
// contents) and writes them to logits_out (nullable).  `logits` is then not
// read.
constexpr int kDecodeFusedLogitCopies = 8;
struct FusedRouter {
    const void *wr;       // [E, H] BF16
    const float *bias;    // [E], nullable
    unsigned long long *ltag;
    float *logits_out;
};
// mxw (nullable): MXFP8 expert weights (FusedMx) instead of wgu/wd (then
// not read); not together with router.  prefetch_inputs: fetch x and the
// logits into L2 while the previous launch drains (device memory only).
cudaError_t launch_decode_fused(const void *x, const float *logits, const void *wgu, const void *wd, int T, int H,
                                int I, int E, int k, int n_sm, float *act, unsigned long long *act_tag,
                                unsigned long long tag_cap, unsigned long long *flags, int32_t *idx_out, float *w_out,
                                float *out, int32_t *exchange_out, unsigned long long wait_ns, int skip_arrival,
                                const FusedRouter *router, const FusedMx *mxw, bool prefetch_inputs,
                                cudaStream_t s);
constexpr unsigned long long kDecodeFusedWaitNs = 2000000000ull;  // default bound of its waits

// moe_ffn_api.cu: an identifier of the calling thread's current CUDA
// context (0 if none can be had), so that per-device set-up is redone in a
// new context, e.g. after cudaDeviceReset.
unsigned long long current_context_id();

// grouped_gemm.cu
cudaError_t gemm_init_device();
bool gemm_supported(int H, int I, int E);
// gate_up reads the chunk's token rows from x [T, H] by perm (row p of the
// sorted order is token perm[p] / k)
cudaError_t launch_gemm_gate_up(const void *x, const int32_t *perm, int k, const void *wgu, const int4 *chunks,
                                const int32_t *nchunks, const int32_t *offs, int n_assign, int H, int I, int E,
                                void *act_hi, void *act_lo, int ctas, cudaStream_t s);
cudaError_t launch_gemm_down(const void *act_hi, const void *act_lo, const void *wd, const int4 *chunks,
                             const int32_t *nchunks, const int32_t *offs, int n_assign, int H, int I, int E, float *z,
                             int ctas, cudaStream_t s);
cudaError_t read_fault_word(uint32_t *flags, bool clear);
// The same two GEMMs with MXFP8 weights: E4M3 codes gq [E, 2I, H] / dq
// [E, H, I] and E8M0 scales gs [E, 2I, mx_scale_bytes(H)] / ds [E, H,
// mx_scale_bytes(I)], converted to exact BF16 tiles inside the kernel.
cudaError_t launch_gemm_gate_up_mx(const void *x, const int32_t *perm, int k, const void *gq, const void *gs,
                                   const int4 *chunks, const int32_t *nchunks, const int32_t *offs, int n_assign, int H,
                                   int I, int E, void *act_hi, void *act_lo, int ctas, cudaStream_t s);
cudaError_t launch_gemm_down_mx(const void *act_hi, const void *act_lo, const void *dq, const void *ds,
                                const int4 *chunks, const int32_t *nchunks, const int32_t *offs, int n_assign, int H,
                                int I, int E, float *z, int ctas, cudaStream_t s);

// Backward pass.  Rows r index the padded sorted order (launch_sort with
// pad 16: each expert's segment rounded up to 16 rows, pad rows zero).
// gate_up_raw: g = W_gate x, u = W_up x [rows][I] FP32.
cudaError_t launch_gemm_gate_up_raw(const void *x, const int32_t *perm, int k, const void *wgu, const int4 *chunks,
                                    const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E,
                                    float *g, float *u, int ctas, cudaStream_t s);
// The forward gate_up GEMM (act as a BF16 hi/lo pair) that also keeps g and
// u [n_rows][I] in FP32 for a later backward pass (the training forward).
cudaError_t launch_gemm_gate_up_keep(const void *x, const int32_t *perm, int k, const void *wgu, const int4 *chunks,
                                     const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E,
                                     void *act_hi, void *act_lo, float *g, float *u, int ctas, cudaStream_t s);
// q = W_down^T dout (dout as ds_hi + ds_lo [rows][H]) and the SwiGLU
// backward: in g, u, w_s; out dgu_hi/lo [rows][2I], wa_hi/lo [rows][I]
// (BF16 pairs) and dwp [rows][I/32] (partial sums of act . q)
struct BwdQOut {
    const float *g, *u, *w_s;
    void *dgu_hi, *dgu_lo, *wa_hi, *wa_lo;
    float *dwp;
};
cudaError_t launch_bwd_q(const void *ds_hi, const void *ds_lo, const void *wd, const int4 *chunks,
                         const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E,
                         const BwdQOut &o, int ctas, cudaStream_t s);
// z [rows][H] = W_gate_up^T (dgu_hi + dgu_lo)
cudaError_t launch_bwd_dx(const void *dgu_hi, const void *dgu_lo, const void *wgu, const int4 *chunks,
                          const int32_t *nchunks, const int32_t *offs, int n_rows, int H, int I, int E, float *z,
                          int ctas, cudaStream_t s);

// grouped_bwd.cu
cudaError_t bwd_init_device();
cudaError_t read_bwd_fault_word(uint32_t *flags, bool clear);
// per padded row: xs = x[token] (BF16), ds_hi/lo = dout[token] split, w_s =
// routing weight; zeros in pad rows
cudaError_t launch_bwd_prep(const void *x, const float *dout, const float *w, const int32_t *perm,
                            const int32_t *offs, int n_rows_max, int E, int H, int k, void *xs, void *ds_hi,
                            void *ds_lo, float *w_s, int n_sm, cudaStream_t s);
// dW_down [E][H][I] = sum_r ds[r] (x) wa[r] over each expert's rows
cudaError_t launch_wgrad_down(const void *ds_hi, const void *ds_lo, const void *wa_hi, const void *wa_lo,
                              const int32_t *offs, const int32_t *counts, int n_rows, int H, int I, int E,
                              float *dwd, int ctas, cudaStream_t s);
// dW_gate_up [E][2I][H] = sum_r dgu[r] (x) xs[r]
cudaError_t launch_wgrad_gate_up(const void *dgu_hi, const void *dgu_lo, const void *xs, const int32_t *offs,
                                 const int32_t *counts, int n_rows, int H, int I, int E, float *dwgu, int ctas,
                                 cudaStream_t s);
// dlogits [T][E] from dwp (I/32 partial sums per row), pos, idx, w
// Zeroes dW_gate_up[e] and dW_down[e] of every expert with counts[e] == 0
// (the weight-gradient kernels skip those experts).
cudaError_t launch_zero_untouched(const int32_t *counts, int E, int H, int I, float *dwgu, float *dwd, int n_sm,
                                  cudaStream_t s);
cudaError_t launch_dlogits(const float *dwp, const int32_t *pos, const int32_t *idx, const float *w, int T, int E,
                           int k, int I, float *dlogits, cudaStream_t s);

}  // namespace moe
