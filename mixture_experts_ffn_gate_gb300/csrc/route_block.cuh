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
// shared memory owned by the warp).  Each lane takes its keys (e = lane +
// 32 i) 8 at a time, sorts them with a sorting network and merges them into
// a sorted list of its kRouteList largest; k rounds then take the warp
// maximum of the list heads (redux on the high, then the low half) and the
// winning lane pops its head.  Larger k rescans the lane's keys below the
// last winner instead.  Lane j < k returns the expert of slot j and its
// softmax weight (the softmax over the k chosen logits, shifted by the
// largest, the logits read back from the winning keys).  With STAGED the
// logits are already in `vals` (the fused decode kernel's router projection
// put them there) and `l` is not read.
constexpr int kRouteList = 8;

__device__ __forceinline__ unsigned long long route_key(float f, int e)
{
    return ((unsigned long long)logit_key(f) << 32) | (uint32_t)~(uint32_t)e;
}

// The float a logit key came from (-0.0 comes back as +0.0, which no
// difference of logits can tell apart).
__device__ __forceinline__ float key_logit(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long v)
{
    const uint32_t hi = (uint32_t)(v >> 32);
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? (uint32_t)v : 0u);
    return ((unsigned long long)mhi << 32) | mlo;
}

// a >= b afterwards
__device__ __forceinline__ void key_order(unsigned long long &a, unsigned long long &b)
{
    const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
}

// 8 keys in descending order: a 19-comparator sorting network of depth 6
__device__ __forceinline__ void sort8_desc(unsigned long long (&x)[8])
{
    key_order(x[0], x[2]); key_order(x[1], x[3]); key_order(x[4], x[6]); key_order(x[5], x[7]);
    key_order(x[0], x[4]); key_order(x[1], x[5]); key_order(x[2], x[6]); key_order(x[3], x[7]);
    key_order(x[0], x[1]); key_order(x[2], x[3]); key_order(x[4], x[5]); key_order(x[6], x[7]);
    key_order(x[2], x[4]); key_order(x[3], x[5]);
    key_order(x[1], x[4]); key_order(x[3], x[6]);
    key_order(x[1], x[2]); key_order(x[3], x[4]); key_order(x[5], x[6]);
}

template <bool STAGED = false>
__device__ __forceinline__ void route_token_warp(const float *__restrict__ l, int E, int k, float *vals, int &sel_j,
                                                 float &w_j)
{
    static_assert(kRouteList == 8, "the sorting network below sorts 8 keys");
    const int lane = threadIdx.x & 31;
    unsigned long long list[kRouteList];
    for (int e0 = 0; e0 < E; e0 += 256) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = e0 + 32 * q + lane;
            if (e < E) v[q] = STAGED ? vals[e] : __ldg(l + e);
        }
        unsigned long long x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = e0 + 32 * q + lane;
            x[q] = e < E ? route_key(v[q], e) : 0ull;
            if (!STAGED && e < E) vals[e] = v[q];
        }
        sort8_desc(x);
        if (e0 == 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q) list[q] = x[q];
        } else {
            // the 8 largest of two descending lists: the larger of each
            // list[q], x[7 - q] pair form a bitonic sequence, sorted by a
            // half-cleaner cascade
#pragma unroll
            for (int q = 0; q < 8; ++q) list[q] = list[q] > x[7 - q] ? list[q] : x[7 - q];
            key_order(list[0], list[4]); key_order(list[1], list[5]);
            key_order(list[2], list[6]); key_order(list[3], list[7]);
            key_order(list[0], list[2]); key_order(list[1], list[3]);
            key_order(list[4], list[6]); key_order(list[5], list[7]);
            key_order(list[0], list[1]); key_order(list[2], list[3]);
            key_order(list[4], list[5]); key_order(list[6], list[7]);
        }
    }
    sel_j = 0;
    uint32_t mine = 0, top = 0;  // logit keys of this lane's slot and of slot 0
    if (k <= kRouteList) {
        for (int r = 0; r < k; ++r) {
            const unsigned long long m = warp_max_key(list[0]);
            if (r == 0) top = (uint32_t)(m >> 32);
            if (lane == r) {
                sel_j = (int)~(uint32_t)m;
                mine = (uint32_t)(m >> 32);
            }
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
            if (r == 0) top = (uint32_t)(m >> 32);
            if (lane == r) {
                sel_j = (int)~(uint32_t)m;
                mine = (uint32_t)(m >> 32);
            }
            if (best == m) {
                best = 0;
                for (int e = lane; e < E; e += 32) {
                    const unsigned long long x = route_key(vals[e], e);
                    if (x < m && x > best) best = x;
                }
            }
        }
    }
    const float ex = lane < k ? expf(key_logit(mine) - key_logit(top)) : 0.0f;
    // a butterfly over the 32 lanes, whose first levels only add the zeros
    // of lanes >= k to lanes < k when k <= 8 (or 16): they are skipped, the
    // sums of lanes < k keep their bits
    float s = ex;
    for (int o = k <= 8 ? 4 : k <= 16 ? 8 : 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
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

}  // namespace moe
