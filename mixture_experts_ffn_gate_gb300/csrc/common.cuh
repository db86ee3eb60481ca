// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Fault bits written to the device fault word when a bounded wait gives up.
enum : uint32_t {
    FAULT_GEMM_PRODUCER = 1u << 0,
    FAULT_GEMM_MMA = 1u << 1,
    FAULT_GEMM_EPILOGUE = 1u << 2,
    FAULT_GEMM_CONVERT = 1u << 3,  // the MXFP8 code converters
};

// 16-byte streaming load that bypasses L1 allocation: expert weights are
// read once per call.
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte read-only load through L1 (activations reused by a block's warps).
__device__ __forceinline__ uint4 ld_nc16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ld_nc_f4(const float *p)
{
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// BF16 pair (low half = element 0) -> two floats, exactly.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Unpack 8 BF16 values held in a uint4.
__device__ __forceinline__ void unpack8(const uint4 &v, float f[8])
{
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// MXFP8 weights (the OCP MX specification's MXFP8: E4M3 codes, one E8M0
// scale per 32 elements along the reduction axis).
// 2^(s - 127) as a float: the biased exponent itself for s >= 1, the
// subnormal 2^-127 for s = 0 (s = 255, NaN in the format, is not an input).
__device__ __forceinline__ float e8m0_scale(uint32_t s)
{
    return __uint_as_float(s ? s << 23 : 0x00400000u);
}

// The FP32 factor 2^(s - 127) of the E8M0 scale s (s = 0 gives the
// subnormal 2^-127; s = 255, NaN in the format, gives +inf).
__device__ __forceinline__ float mx_f32_scale(uint32_t s)
{
    return __uint_as_float(s ? s << 23 : 0x00400000u);
}

// Four E4M3 codes (byte j = element j) times 2^(s - 127) as two BF16 pairs
// (elements 0-1, then 2-3), given f = mx_f32_scale(s): the F16 pair of two
// codes (exact: every E4M3 value is an F16 number), widened to FP32 (exact),
// times f (exact: every product of an E4M3 value and a power of two from
// 2^-127 to 2^127 is an FP32 number or overflows), rounded once to BF16, so
// the result is exact whenever the product is a BF16 number.  The widening
// and the multiplies run on the FMA pipe; an earlier form that moved the F16
// bits into BF16 position with integer masks and shifts and multiplied
// twice in BF16 (the same bits) was bound by the integer pipe and ran the
// grouped MXFP8 GEMMs 8% slower.
__device__ __forceinline__ void e4m3x4_to_bf16x2_f32(uint32_t four_codes, float f, uint32_t &lo, uint32_t &hi)
{
    uint32_t a, b;
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(a), "=r"(b)
        : "r"(four_codes));
    const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&a));
    const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&b));
    const __nv_bfloat162 pa = __floats2bfloat162_rn(fa.x * f, fa.y * f);
    const __nv_bfloat162 pb = __floats2bfloat162_rn(fb.x * f, fb.y * f);
    lo = *reinterpret_cast<const uint32_t *>(&pa);
    hi = *reinterpret_cast<const uint32_t *>(&pb);
}

// 16 E4M3 codes (byte j = element j) to their values in FP32, exactly
// (E4M3 -> F16 -> F32: every E4M3 value is an F16 number).
__device__ __forceinline__ void unpack16_e4m3(const uint4 &v, float (&f)[16])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const __half2_raw r =
                __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] >> (16 * hf)), __NV_E4M3);
            const float2 f2 = __half22float2(__half2(r));
            f[4 * q + 2 * hf] = f2.x;
            f[4 * q + 2 * hf + 1] = f2.y;
        }
}

// Warp sum with a fixed butterfly: every lane ends with the same bits, and
// the association order depends only on the lane layout.
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// warp_sum of N values at once: the same butterfly per value (same bits as
// N calls of warp_sum), with the N shuffle chains interleaved.
template <int N>
__device__ __forceinline__ void warp_sum_n(float (&v)[N])
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int r = 0; r < N; ++r) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
    }
}

// warp_sum of N values (N a power of two <= 32) with the same butterfly, so
// every total has the same bits, but at each of the first log2(N) levels a
// lane keeps half of its values (the upper half if its lane bit for that
// level is set) and receives its partner's copy of that half: N - 1 + 5 -
// log2(N) shuffles instead of 5 N.  Value s ends in lanes
// [s * 32 / N, (s + 1) * 32 / N), each holding the same bits; the return is
// the lane's own total.
template <int N>
__device__ __forceinline__ float warp_sum_split(float (&v)[N], int lane)
{
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
    constexpr int L = N == 1 ? 0 : N == 2 ? 1 : N == 4 ? 2 : N == 8 ? 3 : N == 16 ? 4 : 5;
#pragma unroll
    for (int j = 0; j < L; ++j) {
        const int o = 16 >> j, h = (N >> j) / 2;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 >> L; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// Smallest power of two >= n (n >= 1).
__host__ __device__ constexpr int pow2_ceil(int n) { return n <= 1 ? 1 : 2 * pow2_ceil((n + 1) / 2); }

// silu(g) * u in FP32 with the library expf.
__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// A strict total order on FP32 router logits as an unsigned key: larger
// float -> larger key; -0.0 and +0.0 map to the same key; every NaN maps to
// a fixed key above +inf (NaN logits give a defined, meaningless routing
// instead of broken indices).
__device__ __forceinline__ uint32_t logit_key(float f)
{
    if (f == 0.0f) f = 0.0f;   // -0.0 -> +0.0
    if (f != f) return 0xffffffffu;
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

}  // namespace moe
