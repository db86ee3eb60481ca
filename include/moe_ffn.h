/*
 * moe_ffn.h -- C ABI of libmoeffn.so: the forward and backward passes of a
 * routed Mixture-of-Experts SwiGLU FFN layer on one GB300 GPU (sm_103a).
 *
 * The layer, per token t with activation x[t] (H values) and router logits
 * l[t] (E values):
 *   1. select k experts: k times take the not-yet-chosen expert with the
 *      largest logit, the smaller expert index winning ties (-0.0 == +0.0);
 *      slot j is the j-th pick;
 *   2. w[t][j] = softmax over the k chosen logits;
 *   3. for each slot j, expert e: a = silu(W_gu[e][0:I] x) * (W_gu[e][I:2I] x),
 *      y_j = W_down[e] a   (gate rows 0..I-1, up rows I..2I-1);
 *   4. out[t] = sum over j ascending of w[t][j] * y_j.
 * "Expert routing" and the per-output-dimension FP32 accumulation of the
 * routed experts' contributions are named in the warp-decode article
 * ("Cursor warp decode 공개 ... MoE 추론을 1.84x 가속", section 핵심 내용);
 * keeping the intermediate activation unquantised with BF16 activations and
 * FP32 accumulation is in its section 경쟁 구도 / 비교; a fixed floating-point
 * accumulation order that makes outputs bit-identical regardless of hardware
 * scheduling is in the Mixture-of-Kittens article (asapai.co.kr), section
 * 결정론을 성능과 같은 급으로 올려놓은 선택.
 *
 * Conventions for every call below unless it says otherwise:
 *   - Tensors are row-major and contiguous, in device memory owned by the
 *     caller (e.g. a torch tensor's data_ptr()).  Base pointers must be
 *     16-byte aligned.  BF16 is passed as void* (raw 16-bit patterns).
 *   - x_bf16 [T,H]; router_logits_f32 [T,E]; w_gate_up_bf16 [E,2I,H];
 *     w_down_bf16 [E,H,I]; out_f32 [T,H] (fully overwritten, must not alias
 *     an input).
 *   - Shape limits: T >= 0, 1 <= E <= 1024, 1 <= k <= min(E, 32),
 *     H % 64 == 0, I % 64 == 0, H >= 64, I >= 64; T*k and every index must
 *     fit in int32.  T == 0 returns MOE_OK and enqueues nothing.
 *   - Argument checks are synchronous and happen before anything is
 *     enqueued: a bad argument returns MOE_ERR_INVALID_ARG or
 *     MOE_ERR_UNSUPPORTED_SHAPE and touches no memory.
 *   - Calls are asynchronous on `stream`; results are valid once the stream
 *     reaches the point of the call.  The library keeps no pointer after a
 *     call returns; the caller keeps every buffer alive until the stream's
 *     work is done.
 *   - moe_ffn_forward_ex, moe_ffn_forward_noalloc, moe_ffn_backward (with a
 *     caller workspace) and the training pair may be captured into a CUDA
 *     graph (make one uncaptured call first: it sets up the device);
 *     replays recompute from the captured buffers' current contents.
 *   - Launch failures are returned as MOE_ERR_CUDA (cudaPeekAtLastError);
 *     faults during execution surface at the caller's next synchronisation.
 *   - The fused decode kernel (T <= 4) is launched as a programmatic
 *     dependent (cudaLaunchAttributeProgrammaticStreamSerialization): it
 *     waits for the preceding work on `stream` to complete before it reads
 *     anything, and lets the following launch be scheduled early; a kernel
 *     the caller launches after it with that attribute must, as programmatic
 *     dependent launch requires, call griddepcontrol.wait
 *     (cudaGridDependencySynchronize) before reading this call's outputs.
 *   - Results are deterministic: for the same inputs, path and device the
 *     output bits do not change from run to run or with the launch knobs in
 *     moe_ffn_opts.  The two paths (decode, grouped) are each deterministic
 *     but are not bitwise equal to each other.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* null pointer, negative size, k > E ... */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* valid but outside the shape limits      */
    MOE_ERR_CUDA = 3,              /* a CUDA runtime call or launch failed    */
    MOE_ERR_NO_MEMORY = 4,         /* stream-ordered workspace allocation failed */
    MOE_ERR_WORKSPACE_TOO_SMALL = 5,
    MOE_ERR_TIMEOUT = 6            /* a device-side bounded wait gave up      */
};

/* Execution paths. */
enum {
    MOE_PATH_AUTO = 0,    /* decode for T <= decode_max_tokens, else grouped */
    MOE_PATH_DECODE = 1,  /* warp per output scalar, weights streamed once   */
    MOE_PATH_GROUPED = 2, /* counting sort + tcgen05 grouped GEMMs + combine */
    MOE_PATH_DECODE_FUSED = 3, /* reported only (path_taken): the decode path
                                  for T <= 4 as one kernel that routes the
                                  tokens itself; same results as
                                  MOE_PATH_DECODE */
    MOE_PATH_BACKWARD = 4, /* reported only: moe_ffn_backward's kernels */
    MOE_PATH_TRAIN_FORWARD = 5,  /* reported only: moe_ffn_forward_train   */
    MOE_PATH_TRAIN_BACKWARD = 6  /* reported only: moe_ffn_backward_train  */
};

#define MOE_MAX_STAGES 12

/*
 * Optional knobs and outputs of moe_ffn_forward_ex.  Zero-initialise and set
 * what you need; zero means "library default" for every input field.
 */
typedef struct moe_ffn_opts {
    /* inputs */
    int32_t path;              /* MOE_PATH_AUTO, _DECODE or _GROUPED */
    int32_t decode_max_tokens; /* AUTO threshold on T (default 4) */
    int32_t gate_up_warps;     /* decode gate_up: warps per block, 1..16 (default 8) */
    int32_t down_warps;        /* decode down: warps per block, 1..16 (default 8) */
    int32_t gemm_ctas;         /* grouped GEMMs: persistent CTAs (default: one per SM) */
    /* Test hooks of the fused decode kernel (MOE_PATH_DECODE_FUSED calls
     * only; ignored by the other kernels).  test_wait_limit_us bounds each
     * of its device-side waits (0: 2 s).  test_skip_arrival != 0 makes its
     * last CTA skip its arrival at the grid barrier, so that the barrier's
     * bounded waits run out: the call then writes no output and sets its
     * bit in the device fault word (moe_ffn_device_faults), and the next
     * call on the workspace is correct.  Leave both at zero in production. */
    int32_t test_wait_limit_us;
    int32_t test_skip_arrival;
    int32_t reserved_in[1];    /* must be zero */
    /* nullable: MOE_MAX_STAGES + 1 created events.  When set, the call
     * records stage_events[0] before its first kernel and stage_events[i+1]
     * after kernel i, on `stream`, so the caller can time each kernel with
     * cudaEventElapsedTime.  Under stream capture they are recorded as
     * external event nodes, which time the kernels when the graph replays.
     * Recording events between kernels can change how they overlap, so time
     * whole calls without it. */
    cudaEvent_t *stage_events;
    /* nullable DEVICE int32: a call that takes MOE_PATH_DECODE_FUSED stores
     * (asynchronously, on `stream`) how its CTAs exchanged the act rows:
     * 1 = at a grid barrier (which prepares the workspace's tagged state),
     * 2 = through tagged words, without a barrier.  Other paths leave it. */
    int32_t *exchange_out;
    /* outputs */
    int32_t n_stages;          /* kernels the call enqueued */
    int32_t path_taken;        /* MOE_PATH_DECODE, _DECODE_FUSED or _GROUPED */
    int32_t reserved_out[2];
} moe_ffn_opts;

/*
 * The layer forward pass.  Uses a stream-ordered temporary workspace
 * (cudaMallocAsync / cudaFreeAsync on `stream`), so it is safe on several
 * streams at once, and keeps no state between calls (its decode calls always
 * meet at the grid barrier).  Returns MOE_ERR_NO_MEMORY if that allocation
 * fails.
 */
int moe_ffn_forward(const void *x_bf16, const float *router_logits_f32,
                    const void *w_gate_up_bf16, const void *w_down_bf16,
                    int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                    float *out_f32, cudaStream_t stream);

/*
 * Bytes of device workspace that moe_ffn_forward_ex needs for this shape on
 * either path (the larger of the two), or 0 if the shape is invalid.
 */
size_t moe_ffn_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E,
                               int64_t k);

/*
 * The forward pass with a caller-owned workspace (256-byte aligned, at least
 * moe_ffn_workspace_bytes), optional routing outputs and options.  With a
 * workspace the call allocates nothing and is reentrant; two calls that
 * share a workspace must be ordered on one stream.  The library keeps state in it between calls: the decode path for T <= 4
 * keeps a call counter and tagged scratch at its start.  Calls of any shape
 * may share a workspace (if it is large enough for each): every call lowers
 * the state's record of how much scratch is prepared to what its own other
 * data leave untouched, so a decode call trusts only scratch that no call
 * has overwritten since a barrier call cleared it.  A decode call whose
 * scratch is not prepared meets at a grid barrier and prepares it; the
 * following ones of that shape skip the barrier.  Memory that never served
 * as a workspace needs no initialisation.  Do not write to a workspace
 * between its calls; if its memory holds other data in between (lent to
 * another use, or freed and allocated again), zero its first
 * MOE_FFN_WORKSPACE_STATE_BYTES bytes (e.g. cudaMemsetAsync on `stream`)
 * before its next call, which discards the state.
 *   topk_idx_out  nullable int32 [T,k]: the chosen experts, slot order.
 *   topk_w_out    nullable float [T,k]: their softmax weights.
 *   opts          nullable; see moe_ffn_opts.
 */
#define MOE_FFN_WORKSPACE_STATE_BYTES ((size_t)16384)
int moe_ffn_forward_ex(const void *x_bf16, const float *router_logits_f32,
                       const void *w_gate_up_bf16, const void *w_down_bf16,
                       int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                       float *out_f32, void *workspace, size_t workspace_bytes,
                       int32_t *topk_idx_out, float *topk_w_out,
                       moe_ffn_opts *opts, cudaStream_t stream);

/*
 * The layer with its router projection inside the call: the caller passes
 * the router weights instead of logits.  "Expert routing" is the step the
 * warp-decode article (section 배경 및 맥락) places before the experts; here
 * it is a linear map plus a per-expert bias:
 *   logits[t][e] = round_f32( sum_h x[t][h] * w_router[e][h] + router_bias[e] ),
 * the sum of the BF16 products taken exactly (the GPU forms and accumulates
 * them in FP64, which is exact unless they span more than about 2^40 in
 * magnitude) and rounded once to FP32, so the logits, and the top-k decided
 * on them, are a function of the inputs alone.  Then the layer as in
 * moe_ffn_forward_ex on those logits.
 *   w_router_bf16  [E, H] BF16, one row per expert (a linear layer's weight).
 *   router_bias_f32 nullable [E] FP32 (4-byte aligned).
 *   logits_out     nullable [T, E] FP32: the logits the call computed.
 * Decode calls (the fused decode kernel, T <= 4) compute the logits inside
 * that kernel, each CTA a share, exchanged between CTAs through the
 * workspace: no separate router launch.  Other calls run one router kernel
 * first.  The FP64 rate of the GPU makes that kernel slow for large T (at
 * T = 2048, E = 256, H = 6144 it takes milliseconds): batches of that size
 * are better served by logits from the caller's own GEMM and
 * moe_ffn_forward_ex.  The workspace (at least
 * moe_ffn_router_workspace_bytes) is moe_ffn_forward_ex's, with the same
 * state and rules, plus room for the logits.
 */
size_t moe_ffn_router_workspace_bytes(int64_t T, int64_t H, int64_t I,
                                      int64_t E, int64_t k);
int moe_ffn_forward_router(const void *x_bf16, const void *w_router_bf16,
                           const float *router_bias_f32,
                           const void *w_gate_up_bf16, const void *w_down_bf16,
                           int64_t T, int64_t H, int64_t I, int64_t E,
                           int64_t k, float *out_f32, void *workspace,
                           size_t workspace_bytes, float *logits_out,
                           int32_t *topk_idx_out, float *topk_w_out,
                           moe_ffn_opts *opts, cudaStream_t stream);

/*
 * The layer with MXFP8 expert weights.  The Mixture-of-Kittens article ("커서가 MoE 학습 메가커널 믹스처 오브
 * 키튼스를 아파치 2.0으로 공개했다", section 2.37배는 어떤 기준선과 비교한
 * 숫자인가) measures the layer with MXFP8 operands; the format is the OCP
 * Microscaling (MX) specification's MXFP8 with E4M3 elements, applied here
 * to the expert weights (the activations stay BF16):
 *   w_gate_up_e4m3  [E, 2I, H] uint8 E4M3 codes (row layout as for BF16),
 *   w_gate_up_scale [E, 2I, Sh] uint8 E8M0 scales, Sh = MOE_FFN_MX_SCALE_BYTES(H),
 *   w_down_e4m3     [E, H, I] uint8 E4M3 codes,
 *   w_down_scale    [E, H, Si] uint8 E8M0 scales, Si = MOE_FFN_MX_SCALE_BYTES(I).
 * Weight [e, r, c] = E4M3(code) * 2^(scale[e, r, c / 32] - 127); a scale row
 * holds K / 32 scales, then padding to a multiple of 16 bytes (ignored).
 * NaN codes (E4M3 S.1111.111, scale 255) are not valid inputs.  Products
 * and sums are formed in FP32 as in the BF16 path; the results are within
 * the same tolerance of the FP64 layer on the dequantised weights.
 * All device pointers 16-byte aligned; the workspace is moe_ffn_forward_ex's
 * (at least moe_ffn_workspace_bytes, same state rules).  Paths (path_taken
 * tells which): AUTO takes the fused decode kernel for T <= 4 where it fits,
 * the general decode kernels up to T = 8 (opts->decode_max_tokens moves
 * this bound) and the grouped tensor-core GEMMs beyond, which load the E4M3
 * code tiles and convert
 * them to exact BF16 tiles (each weight a BF16 number whenever its value is
 * in BF16's range) in shared memory before their BF16 MMAs.  opts->path
 * DECODE forces the decode kernels, which take at most 64 tokens (larger T
 * returns MOE_ERR_UNSUPPORTED_SHAPE, with nothing launched); GROUPED forces
 * the grouped path.
 */
#define MOE_FFN_MX_SCALE_BYTES(K) ((((K) / 32) + 15) / 16 * 16)
int moe_ffn_forward_mxfp8(const void *x_bf16, const float *router_logits_f32,
                          const void *w_gate_up_e4m3, const void *w_gate_up_scale,
                          const void *w_down_e4m3, const void *w_down_scale,
                          int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                          float *out_f32, void *workspace,
                          size_t workspace_bytes, int32_t *topk_idx_out,
                          float *topk_w_out, moe_ffn_opts *opts,
                          cudaStream_t stream);

/*
 * End-to-end form for callers whose tokens live in host memory: x_host
 * [T,H] bf16, logits_host [T,E] f32 and out_host [T,H] f32 are HOST buffers
 * (page-locked for the copies to be asynchronous); the weights are device
 * buffers as above.  The call enqueues host->device copies of the inputs,
 * the forward pass and the device->host copy of the output on `stream`;
 * out_host is valid after the stream is synchronised.  The workspace
 * (device, at least moe_ffn_host_workspace_bytes) also holds the staged
 * inputs and output, and keeps the same state, under the same rules, as
 * moe_ffn_forward_ex's.  When the three host buffers are page-locked and mapped
 * (cudaHostAlloc, cudaMallocHost, torch's pin_memory), 16-byte aligned and
 * at most 1 MiB together, the kernels read the inputs and write the output
 * in place through the host link instead (no separate copies; same
 * results); the caller must not touch them until the stream reaches the
 * end of the call.
 */
size_t moe_ffn_host_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E,
                                    int64_t k);
int moe_ffn_forward_host(const void *x_host, const float *logits_host,
                         const void *w_gate_up_bf16, const void *w_down_bf16,
                         int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                         float *out_host, void *workspace,
                         size_t workspace_bytes, moe_ffn_opts *opts,
                         cudaStream_t stream);

/*
 * No counterpart in the pages: an entry point for callers that cannot
 * allocate device memory once they are running -- a serving loop whose
 * latency budget cannot absorb an allocation that may synchronise the device
 * or fail under memory pressure, or a plugin whose host engine owns all
 * device memory through its own pool.  Same arguments, path choice and
 * results as moe_ffn_forward, but the scratch lives in a fixed device array
 * of MOE_FFN_NOALLOC_SCRATCH_BYTES inside the library (present in every GPU
 * context that loads the library, until the process exits); the call
 * allocates nothing.  Shapes whose workspace (moe_ffn_workspace_bytes)
 * exceeds that size return MOE_ERR_WORKSPACE_TOO_SMALL before anything is
 * enqueued.  The first call on each device looks up the array's device
 * address (set-up, once per device, with that device current, and again if
 * the device's context changes, e.g. after cudaDeviceReset); make that
 * first call before any stream capture.  All calls share the array: calls
 * whose GPU work overlaps (other streams, unordered host threads) race and
 * return wrong results, so order them on one stream.  The array serves as
 * the workspace of moe_ffn_forward_ex, with the state that keeps between
 * calls.
 */
#define MOE_FFN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int moe_ffn_forward_noalloc(const void *x_bf16, const float *router_logits_f32,
                            const void *w_gate_up_bf16, const void *w_down_bf16,
                            int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                            float *out_f32, cudaStream_t stream);

/*
 * The backward pass of the layer (the Mixture-of-Kittens article,
 * asapai.co.kr, section 2.37배는 어떤 기준선과 비교한 숫자인가, measures the
 * layer's forward and backward passes in training; the gradients below are
 * the chain rule of the forward definition at the top of this file).  For
 * the upstream gradient dout_f32 [T,H] = dL/dout, with the routing of the
 * forward pass recomputed from the logits (same selection and weights):
 *   q = W_down[e]^T dout[t],  dw_j = a . q,  da = w_j q,
 *   dg = da u s (1 + g (1 - s)),  du = da g s      (s = sigmoid(g));
 *   dx_f32 [T,H]          = sum_j W_gate[e]^T dg + W_up[e]^T du
 *   dlogits_f32 [T,E]     = w_j (dw_j - sum_m w_m dw_m) at the selected
 *                           experts s_j, 0 elsewhere (the selection is
 *                           piecewise constant in the logits)
 *   dw_gate_up_f32 [E,2I,H] = sum over e's assignments of [dg ; du] x[t]^T
 *   dw_down_f32 [E,H,I]   = sum over e's assignments of (w_j dout[t]) a^T
 * All four outputs are fully overwritten (experts no token selects get
 * zeros) and must not alias each other or an input.  Arithmetic: BF16
 * inputs, FP32 accumulation, FP32 intermediates; tensor-core products take
 * FP32 operands as BF16 hi + lo pairs.  Deterministic (no floating-point
 * atomics): the same inputs give the same output bits on every run.
 * Same shape limits and pointer rules as the forward pass; the call runs
 * the grouped tensor-core kernels for every T (opts->path AUTO or GROUPED,
 * else MOE_ERR_UNSUPPORTED_SHAPE).  workspace: device, 256-byte aligned, at
 * least moe_ffn_backward_workspace_bytes; NULL makes the call allocate one
 * stream-ordered (cudaMallocAsync / cudaFreeAsync on `stream`).  The
 * workspace may be one that forward calls also use: the backward call
 * keeps the fused decode kernel's state words valid (it marks the state's
 * tag region as spent).  T == 0 zeroes the two weight gradients
 * (cudaMemsetAsync) and returns.  opts (nullable): gemm_ctas and
 * stage_events as for the forward pass; path_taken = MOE_PATH_BACKWARD.
 */
size_t moe_ffn_backward_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E,
                                        int64_t k);
int moe_ffn_backward(const void *x_bf16, const float *router_logits_f32,
                     const void *w_gate_up_bf16, const void *w_down_bf16,
                     const float *dout_f32, int64_t T, int64_t H, int64_t I,
                     int64_t E, int64_t k, float *dx_f32, float *dlogits_f32,
                     float *dw_gate_up_f32, float *dw_down_f32, void *workspace,
                     size_t workspace_bytes, moe_ffn_opts *opts,
                     cudaStream_t stream);

/*
 * The training pair: a forward pass that keeps, in a caller-owned state
 * buffer, the gate/up projections the backward pass needs, and the backward
 * pass that reads them instead of recomputing them (which re-reads every
 * touched expert's W_gate_up).  The layer and the gradients are those of
 * moe_ffn_forward and moe_ffn_backward (same definitions), with the same
 * bits:
 *   - moe_ffn_forward_train's out equals moe_ffn_forward_ex's on the
 *     grouped path (opts->path = MOE_PATH_GROUPED) bit for bit;
 *   - moe_ffn_backward_train's four gradients equal moe_ffn_backward's on
 *     the same inputs bit for bit.
 * state: device, 256-byte aligned, at least moe_ffn_train_state_bytes
 * (= moe_ffn_backward_workspace_bytes) for the call's T, H, I, E, k; the
 * forward call leaves in it g = W_gate x and u = W_up x in FP32 for every
 * assignment, in the order of the assignments sorted by expert (each
 * expert's segment rounded up to 16 rows); the rest is scratch space of
 * either call.  Call order on the stream: moe_ffn_forward_train, then
 * moe_ffn_backward_train with the same x, logits, weights and shape, and
 * nothing else writing to the state in between (a plain forward or
 * backward call given the state as its workspace overwrites it).  The
 * backward call routes and sorts the logits again (two small kernels) and
 * reads only g and u from the state, never writing them, so it may run
 * again on one state (for another dout), and a state from another call
 * gives wrong gradients but no access outside the call's own buffers.
 * Both run the grouped tensor-core kernels for every T (opts->path AUTO or
 * GROUPED, else MOE_ERR_UNSUPPORTED_SHAPE); same shape limits, pointer
 * rules and statuses as moe_ffn_backward; opts (nullable): gemm_ctas and
 * stage_events; path_taken = MOE_PATH_TRAIN_FORWARD / _TRAIN_BACKWARD.
 * T == 0: the forward call does nothing; the backward call zeroes the two
 * weight gradients (cudaMemsetAsync).
 */
size_t moe_ffn_train_state_bytes(int64_t T, int64_t H, int64_t I, int64_t E,
                                 int64_t k);
int moe_ffn_forward_train(const void *x_bf16, const float *router_logits_f32,
                          const void *w_gate_up_bf16, const void *w_down_bf16,
                          int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                          float *out_f32, void *state, size_t state_bytes,
                          moe_ffn_opts *opts, cudaStream_t stream);
int moe_ffn_backward_train(const void *x_bf16, const float *router_logits_f32,
                           const void *w_gate_up_bf16, const void *w_down_bf16,
                           const float *dout_f32, int64_t T, int64_t H, int64_t I,
                           int64_t E, int64_t k, float *dx_f32, float *dlogits_f32,
                           float *dw_gate_up_f32, float *dw_down_f32, void *state,
                           size_t state_bytes, moe_ffn_opts *opts,
                           cudaStream_t stream);

/* Static text for a status code. */
const char *moe_ffn_status_string(int status);

/* Name of kernel `stage` (0-based) on `path`, or NULL past the last one. */
const char *moe_ffn_stage_name(int path, int stage);

/*
 * Device fault word: bit flags that kernels set when a bounded device-side
 * wait gives up (instead of hanging): bits 0-7 the grouped GEMMs, 8-15 the
 * fused decode kernel, 16-23 the backward pass's weight-gradient GEMMs.
 * Reads the current device's word
 * synchronously into *flags and, if clear != 0, resets it.  Returns MOE_OK,
 * or MOE_ERR_CUDA if the read fails.  A non-zero word means some call since
 * the last clear returned garbage in out_f32.
 */
int moe_ffn_device_faults(uint32_t *flags, int clear);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
