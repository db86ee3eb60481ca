// kernels.h -- launchers of the library's kernels (internal to libmoeffn.so).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Grouped path: at most this many assignments (token rows) per GEMM N-chunk.
constexpr int kGemmChunkMax = 64;

// routing.cu
cudaError_t routing_init_device();
cudaError_t launch_router(const float *logits, int T, int E, int k, int32_t *idx, float *w, int32_t *idx_copy,
                          float *w_copy, cudaStream_t s);
size_t sort_smem_bytes(int E);
cudaError_t launch_sort(const int32_t *idx, int n_assign, int E, int chunk_max, int32_t *offs, int32_t *perm,
                        int32_t *pos, int32_t *uexp, int32_t *ucount, int4 *chunks, int32_t *nchunks,
                        cudaStream_t s);
cudaError_t launch_gather(const void *x, const int32_t *perm, int k, int H, int n_rows, void *xs, int n_sm,
                          cudaStream_t s);
cudaError_t launch_combine(const float *z, const float *w, const int32_t *pos, int T, int H, int k, float *out,
                           int n_sm, cudaStream_t s);

// decode.cu
cudaError_t decode_init_device();
int decode_down_tok_tile(int T, int k);
cudaError_t launch_decode_gate_up(const void *x, const void *wgu, const int32_t *uexp, const int32_t *ucount,
                                  const int32_t *offs, const int32_t *perm, int T, int H, int I, int E, int k,
                                  int warps, float *act, cudaStream_t s);
cudaError_t launch_decode_down(const float *act, const void *wd, const float *w, const int32_t *uexp,
                               const int32_t *ucount, const int32_t *offs, const int32_t *perm, int T, int H,
                               int I, int k, int warps, float *out, cudaStream_t s);

// decode_fused.cu: a decode step of up to four tokens in one cooperative
// kernel.  act: [T*k][I] FP32 scratch; flags: kDecodeFusedFlagWords 64-bit
// words and act_tag: decode_fused_tag_words(k, I) 64-bit words, both kept by
// the kernel between calls (any initial contents) and written by nothing
// else; act_tag may be null (every call then meets at a grid barrier).
constexpr int kMaxGridCtas = 1024;
constexpr int kDecodeFusedFlagWords = kMaxGridCtas + 32;
cudaError_t decode_fused_init_device();
cudaError_t read_decode_fused_fault_word(uint32_t *flags, bool clear);
bool decode_fused_supported(int T, int H, int I, int E, int k, int n_sm);
size_t decode_fused_tag_words(int k, int I);
cudaError_t launch_decode_fused(const void *x, const float *logits, const void *wgu, const void *wd, int T, int H,
                                int I, int E, int k, int n_sm, float *act, unsigned long long *act_tag,
                                unsigned long long *flags, int32_t *idx_out, float *w_out, float *out,
                                cudaStream_t s);

// grouped_gemm.cu
cudaError_t gemm_init_device();
bool gemm_supported(int H, int I, int E);
cudaError_t launch_gemm_gate_up(const void *xs, const void *wgu, const int4 *chunks, const int32_t *nchunks,
                                const int32_t *offs, int n_assign, int H, int I, int E, void *act_hi, void *act_lo,
                                int ctas, cudaStream_t s);
cudaError_t launch_gemm_down(const void *act_hi, const void *act_lo, const void *wd, const int4 *chunks,
                             const int32_t *nchunks, const int32_t *offs, int n_assign, int H, int I, int E, float *z,
                             int ctas, cudaStream_t s);
cudaError_t read_fault_word(uint32_t *flags, bool clear);

}  // namespace moe
