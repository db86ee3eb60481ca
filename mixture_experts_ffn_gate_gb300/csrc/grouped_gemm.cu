// grouped_gemm.cu -- the large-T path's grouped GEMMs (tcgen05, TMEM, TMA).
#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ uint32_t g_fault_word = 0;

cudaError_t read_fault_word(uint32_t *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_fault_word, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(uint32_t));
}

cudaError_t gemm_init_device() { return cudaSuccess; }

bool gemm_supported(int, int) { return false; }

cudaError_t launch_gemm_gate_up(const void *, const void *, const int4 *, const int32_t *, int, int, int, int, void *,
                                void *, int, cudaStream_t)
{
    return cudaErrorNotSupported;
}

cudaError_t launch_gemm_down(const void *, const void *, const void *, const int4 *, const int32_t *, int, int, int,
                             int, float *, int, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace moe
