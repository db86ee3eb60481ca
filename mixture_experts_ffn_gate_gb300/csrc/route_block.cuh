// route_block.cuh -- top-k selection and softmax weights for one token,
// computed by one warp.  Used by the router kernel and by the fused decode
// kernel, which routes its tokens itself; both give the same bits.
#pragma once

#include "common.cuh"

namespace moe {

// One warp routes one token under a strict total order -- a larger logit
// first, on equal logits the smaller index (-0.0 == +0.0).  The key of
// expert e is the 64-bit (logit_key << 32) | ~e: keys are unique and 0 lies
// below every key.  The warp copies the E logits into `vals` (E words of
// shared memory owned by the warp, eight loads in flight per lane).  For
// k <= kRouteList each lane keeps the kRouteList largest of its own keys
// (e = lane + 32 i) in a sorted register list; k rounds then take the warp
// maximum of the list heads (redux on the high, then the low half) and the
// winning lane pops its head.  Larger k rescans the lane's keys below the
// last winner instead.  Lane j < k returns the expert of slot j and its
// softmax weight (the softmax over the k chosen logits, shifted by the
// largest).  With STAGED the logits are already in `vals` (the fused decode
// kernel's router projection put them there) and `l` is not read.
constexpr int kRouteList = 8;

__device__ __forceinline__ unsigned long long route_key(float f, int e)
{
    return ((unsigned long long)logit_key(f) << 32) | (uint32_t)~(uint32_t)e;
}

__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long v)
{
    const uint32_t hi = (uint32_t)(v >> 32);
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? (uint32_t)v : 0u);
    return ((unsigned long long)mhi << 32) | mlo;
}

template <bool STAGED = false>
__device__ __forceinline__ void route_token_warp(const float *__restrict__ l, int E, int k, float *vals, int &sel_j,
                                                 float &w_j)
{
    const int lane = threadIdx.x & 31;
    unsigned long long list[kRouteList];
#pragma unroll
    for (int q = 0; q < kRouteList; ++q) list[q] = 0;
    for (int e0 = 0; e0 < E; e0 += 256) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = e0 + 32 * q + lane;
            if (e < E) v[q] = STAGED ? vals[e] : __ldg(l + e);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = e0 + 32 * q + lane;
            if (e < E) {
                if (!STAGED) vals[e] = v[q];
                // insert into the descending list: new[i] = max(old[i], min(old[i-1], x))
                const unsigned long long x = route_key(v[q], e);
#pragma unroll
                for (int i = kRouteList - 1; i > 0; --i) {
                    const unsigned long long m = list[i - 1] < x ? list[i - 1] : x;
                    list[i] = list[i] > m ? list[i] : m;
                }
                list[0] = list[0] > x ? list[0] : x;
            }
        }
    }
    sel_j = 0;
    if (k <= kRouteList) {
        for (int r = 0; r < k; ++r) {
            const unsigned long long m = warp_max_key(list[0]);
            if (lane == r) sel_j = (int)~(uint32_t)m;
            if (list[0] == m) {
#pragma unroll
                for (int i = 0; i < kRouteList - 1; ++i) list[i] = list[i + 1];
                list[kRouteList - 1] = 0;
            }
        }
    } else {
        unsigned long long best = list[0];
        for (int r = 0; r < k; ++r) {
            const unsigned long long m = warp_max_key(best);
            if (lane == r) sel_j = (int)~(uint32_t)m;
            if (best == m) {
                best = 0;
                for (int e = lane; e < E; e += 32) {
                    const unsigned long long x = route_key(vals[e], e);
                    if (x < m && x > best) best = x;
                }
            }
        }
    }
    __syncwarp();
    const float l0 = vals[__shfl_sync(0xffffffffu, sel_j, 0)];
    const float ex = lane < k ? expf(vals[sel_j] - l0) : 0.0f;
    const float s = warp_sum(ex);
    w_j = lane < k ? ex / s : 0.0f;
}

// The router projection sum_h x[h] * w[h] + bias, rounded once to FP32,
// computed in 256-element slices so that several warps can share one logit.
// Slice s holds elements [256 s, 256 s + 256); lane l takes the 8 at
// 256 s + 8 l.  Each product of two BF16 values is exact in FP32 (unless its
// magnitude is below 2^-133); the 8 products are summed pairwise in FP64 and
// the lanes' sums by a fixed FP64 butterfly (router_slice_warp).  The logit
// is the sum of the slices in ascending order, plus the bias, rounded once
// to FP32 (router_logit_sum).  FP64 holds these sums exactly unless the
// products span more than about 2^40 in magnitude, so the logit is the
// exact sum rounded once; either way every router logit the library
// computes follows this one order and has the same bits.
// x, w: BF16 rows in global memory, 16-byte aligned, H a multiple of 8.
__device__ __forceinline__ double router_slice_warp(const uint16_t *x, const uint16_t *__restrict__ w, int H, int s,
                                                    int lane)
{
    const int h = 256 * s + 8 * lane;
    double d = 0.0;
    if (h < H) {
        float wf[8], xf[8];
        unpack8(ld_stream16(w + h), wf);
        unpack8(ld_nc16(x + h), xf);
        double p[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) p[q] = (double)(wf[q] * xf[q]);
        d = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    return d;
}

__host__ __device__ constexpr int router_slices(int H) { return (H + 255) / 256; }

__device__ __forceinline__ float router_logit_sum(const double *slice, int ns, float bias)
{
    double acc = 0.0;
    for (int s = 0; s < ns; ++s) acc += slice[s];
    return __double2float_rn(acc + (double)bias);
}

// One router logit by one warp (all its slices in turn, the same order).
__device__ __forceinline__ float router_logit_warp(const uint16_t *x, const uint16_t *__restrict__ w, int H,
                                                   float bias, int lane)
{
    double acc = 0.0;
    for (int s = 0; s < router_slices(H); ++s) acc += router_slice_warp(x, w, H, s, lane);
    return __double2float_rn(acc + (double)bias);
}

// Block-wide form: warp 0 routes, every thread of the block must call this;
// vals: E words of shared memory; sel[k] and w[k] (shared) receive the chosen
// experts in slot order and their softmax weights.
__device__ __forceinline__ void route_token_block(const float *__restrict__ l, int E, int k, float *vals, int *sel,
                                                  float *w)
{
    if (threadIdx.x < 32) {
        int e;
        float wt;
        route_token_warp(l, E, k, vals, e, wt);
        if (threadIdx.x < k) {
            sel[threadIdx.x] = e;
            w[threadIdx.x] = wt;
        }
    }
    __syncthreads();
}

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the next grid to be scheduled.  No-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace moe
