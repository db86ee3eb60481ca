// route_block.cuh -- top-k selection and softmax weights for one token,
// computed by a whole thread block.  Used by the router kernel and by the
// single-token decode kernels, which route their token themselves; both give
// the same bits.
#pragma once

#include "common.cuh"

namespace moe {

// Every thread of the block must call this.  keys: E x 8 bytes of shared
// memory; sel[k] and w[k] (shared) receive the chosen experts in slot order
// and their softmax weights.  Ranking uses a strict total order (larger
// logit first, the smaller index on ties, -0.0 == +0.0), so the ranks below
// k are exactly the k slots.
__device__ __forceinline__ void route_token_block(const float *__restrict__ l, int E, int k,
                                                  unsigned long long *keys, int *sel, float *w)
{
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        keys[e] = ((unsigned long long)logit_key(__ldg(l + e)) << 32) | (uint32_t)(0xffffffffu - (uint32_t)e);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const unsigned long long me = keys[e];
        int r = 0;
        for (int j = 0; j < E; ++j) r += keys[j] > me;
        if (r < k) sel[r] = e;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const float l0 = __ldg(l + sel[0]);
        const float ex = lane < k ? expf(__ldg(l + sel[lane]) - l0) : 0.0f;
        const float s = warp_sum(ex);
        if (lane < k) w[lane] = ex / s;
    }
    __syncthreads();
}

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the next grid to be scheduled.  No-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace moe
