// decode.cu -- the small-T path: one warp per output scalar, each touched
// expert's weights streamed from HBM once, FP32 everywhere after the BF16
// loads.
//
// The warp-decode article ("Cursor warp decode 공개 ... MoE 추론을 1.84x
// 가속", section 핵심 내용) describes two kernels whose warps each own one
// neuron (gate/up) or one output dimension (down) and add the routed
// experts' contributions into FP32 directly, with no padding, scatter or
// per-expert output buffers; its section 경쟁 구도 / 비교 drops the
// intermediate activation quantisation.  This file keeps those properties:
//   gate_up: warp per (touched expert, neuron i); loads gate row i and up row
//            I+i with 128-bit streaming loads, dots them with every token the
//            expert serves, reduces with a fixed shuffle butterfly and writes
//            silu(g)*u in FP32 (act[assignment, i]).
//   down:    block per group of DOWN_HW output dims; its warps walk the
//            touched experts, dot each W_down row with the FP32 activations
//            of that expert's tokens, park the per-assignment partials in
//            shared memory, then sum each token's k partials in slot order.
// Every output's arithmetic (lane split, chunk order, butterfly, slot order)
// is independent of the launch shape, so the bits do not change with the
// warps-per-block knobs.
//
// MX instantiations take MXFP8 weights (E4M3 codes, one E8M0 scale per 32
// elements along the reduction axis): a lane reads 16 codes per step,
// converts them to FP32 exactly, forms the partial sum with the FP32
// activations and adds it times the block's power-of-two scale, as the fused
// kernel's MX instantiation does.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int GU_UNR = 4;  // 256-element chunks in flight per lane
constexpr int DOWN_HW = 4; // output dims per block in down
constexpr int DOWN_UNR = 2;
constexpr int MX_UNR = 2;   // 512-element steps in flight per lane (MXFP8 rows)

// MXFP8 weights of a call: codes gq [E][2I][H], dq [E][H][I]; scales gs
// [E][2I][hs], ds [E][H][is] (hs, is: scale bytes per row).
struct DecodeMx {
    const uint8_t *gq, *gs, *dq, *ds;
    int hs, is;
};

// GU_TB: assignments (tokens of one expert) per pass; at most T.
template <int GU_TB, bool MX>
__global__ void __launch_bounds__(512) decode_gate_up_kernel(const uint16_t *__restrict__ x,
                                                              const uint16_t *__restrict__ wgu,
                                                              const int32_t *__restrict__ uexp,
                                                              const int32_t *__restrict__ ucount,
                                                              const int32_t *__restrict__ offs,
                                                              const int32_t *__restrict__ perm, int H, int I,
                                                              int k, float *__restrict__ act, DecodeMx mx)
{
    const int s = blockIdx.y;
    if (s >= *ucount) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = blockIdx.x * (blockDim.x >> 5) + warp;
    if (i >= I) return;
    const int e = uexp[s];
    const int a0 = offs[e], n = offs[e + 1] - a0;
    const uint16_t *gate = wgu + ((int64_t)e * 2 * I + i) * H;
    const uint16_t *up = gate + (int64_t)I * H;

    for (int p0 = 0; p0 < n; p0 += GU_TB) {
        const int nb = min(GU_TB, n - p0);
        int arow[GU_TB];
        const uint16_t *xr[GU_TB];
#pragma unroll
        for (int b = 0; b < GU_TB; ++b) {
            arow[b] = perm[a0 + p0 + min(b, nb - 1)];
            xr[b] = x + (int64_t)(arow[b] / k) * H;
        }
        float g[GU_TB], u[GU_TB];
#pragma unroll
        for (int b = 0; b < GU_TB; ++b) g[b] = u[b] = 0.0f;

        if constexpr (MX) {
            const int64_t r0 = (int64_t)e * 2 * I + i;  // gate row; up row r0 + I
            const uint8_t *gq = mx.gq + r0 * H, *uq = gq + (int64_t)I * H;
            const uint8_t *gs = mx.gs + r0 * mx.hs, *us = gs + (int64_t)I * mx.hs;
            for (int h = lane * 16; h < H; h += 512 * MX_UNR) {
                uint4 gw[MX_UNR], uw[MX_UNR];
                float sg[MX_UNR], su[MX_UNR];
#pragma unroll
                for (int q = 0; q < MX_UNR; ++q) {
                    const int hq = h + q * 512;
                    if (hq < H) {
                        gw[q] = ld_stream16(gq + hq);
                        uw[q] = ld_stream16(uq + hq);
                        sg[q] = e8m0_scale(__ldg(gs + (hq >> 5)));
                        su[q] = e8m0_scale(__ldg(us + (hq >> 5)));
                    }
                }
#pragma unroll
                for (int q = 0; q < MX_UNR; ++q) {
                    const int hq = h + q * 512;
                    if (hq < H) {
                        float gf[16], uf[16];
                        unpack16_e4m3(gw[q], gf);
                        unpack16_e4m3(uw[q], uf);
#pragma unroll
                        for (int b = 0; b < GU_TB; ++b) {
                            if (b < nb) {
                                float xf[16];
                                unpack8(ld_nc16(xr[b] + hq), xf);
                                unpack8(ld_nc16(xr[b] + hq + 8), xf + 8);
                                float pg = 0.0f, pu = 0.0f;
#pragma unroll
                                for (int c = 0; c < 16; ++c) {
                                    pg = fmaf(gf[c], xf[c], pg);
                                    pu = fmaf(uf[c], xf[c], pu);
                                }
                                g[b] = fmaf(pg, sg[q], g[b]);
                                u[b] = fmaf(pu, su[q], u[b]);
                            }
                        }
                    }
                }
            }
        } else {
        for (int h = lane * 8; h < H; h += 256 * GU_UNR) {
            uint4 gw[GU_UNR], uw[GU_UNR];
#pragma unroll
            for (int q = 0; q < GU_UNR; ++q) {
                const int hq = h + q * 256;
                if (hq < H) {
                    gw[q] = ld_stream16(gate + hq);
                    uw[q] = ld_stream16(up + hq);
                }
            }
#pragma unroll
            for (int q = 0; q < GU_UNR; ++q) {
                const int hq = h + q * 256;
                if (hq < H) {
                    float gf[8], uf[8];
                    unpack8(gw[q], gf);
                    unpack8(uw[q], uf);
#pragma unroll
                    for (int b = 0; b < GU_TB; ++b) {
                        if (b < nb) {
                            float xf[8];
                            unpack8(ld_nc16(xr[b] + hq), xf);
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                g[b] = fmaf(gf[c], xf[c], g[b]);
                                u[b] = fmaf(uf[c], xf[c], u[b]);
                            }
                        }
                    }
                }
            }
        }
        }
#pragma unroll
        for (int b = 0; b < GU_TB; ++b) {
            if (b < nb) {
                const float gs = warp_sum(g[b]);
                const float us = warp_sum(u[b]);
                if (lane == 0) act[(int64_t)arow[b] * I + i] = swiglu(gs, us);
            }
        }
    }
}

// First index in perm[lo, hi) whose token (perm / k) is >= t; the tokens of
// one expert's segment are ascending.
__device__ __forceinline__ int lower_bound_token(const int32_t *perm, int lo, int hi, int k, int t)
{
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (perm[mid] / k < t) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Block (blockIdx.x = group of DOWN_HW output dims, blockIdx.y = tile of
// tok_tile tokens).  part[hw][(t - t0)*k + j] holds W_down[e_j, h0+hw, :] .
// act[t*k+j, :] for the tile's tokens.  DOWN_TB: assignments per pass.
template <int DOWN_TB, bool MX>
__global__ void __launch_bounds__(512) decode_down_kernel(const float *__restrict__ act,
                                                           const uint16_t *__restrict__ wd,
                                                           const float *__restrict__ wts,
                                                           const int32_t *__restrict__ uexp,
                                                           const int32_t *__restrict__ ucount,
                                                           const int32_t *__restrict__ offs,
                                                           const int32_t *__restrict__ perm, int T, int H, int I,
                                                           int k, int tok_tile, float *__restrict__ out, DecodeMx mx)
{
    extern __shared__ float part[];  // [DOWN_HW][tok_tile * k]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int h0 = blockIdx.x * DOWN_HW;
    const int t0 = blockIdx.y * tok_tile;
    const int t1 = min(T, t0 + tok_tile);
    const int span = tok_tile * k;
    const int U = *ucount;
    const int a_lo = t0 * k;  // assignment ids of the tile are [t0*k, t1*k)

    for (int s = warp; s < U; s += nwarps) {
        const int e = uexp[s];
        const int seg0 = offs[e], seg1 = offs[e + 1];
        const int p_begin = (t0 == 0) ? seg0 : lower_bound_token(perm, seg0, seg1, k, t0);
        const int p_end = (t1 == T) ? seg1 : lower_bound_token(perm, p_begin, seg1, k, t1);
        if (p_begin >= p_end) continue;
        const uint16_t *wrow = wd + ((int64_t)e * H + h0) * I;

        for (int p0 = p_begin; p0 < p_end; p0 += DOWN_TB) {
            const int nb = min(DOWN_TB, p_end - p0);
            int arow[DOWN_TB];
#pragma unroll
            for (int b = 0; b < DOWN_TB; ++b) arow[b] = perm[p0 + min(b, nb - 1)];
            float acc[DOWN_HW][DOWN_TB];
#pragma unroll
            for (int r = 0; r < DOWN_HW; ++r)
#pragma unroll
                for (int b = 0; b < DOWN_TB; ++b) acc[r][b] = 0.0f;

            if constexpr (MX) {
                const int64_t r0 = (int64_t)e * H + h0;
                const uint8_t *wq = mx.dq + r0 * I, *ws = mx.ds + r0 * mx.is;
                for (int c = lane * 16; c < I; c += 512 * MX_UNR) {
                    uint4 wv[MX_UNR][DOWN_HW];
                    float sc[MX_UNR][DOWN_HW];
#pragma unroll
                    for (int q = 0; q < MX_UNR; ++q) {
                        const int cq = c + q * 512;
                        if (cq < I) {
#pragma unroll
                            for (int r = 0; r < DOWN_HW; ++r) {
                                wv[q][r] = ld_stream16(wq + (int64_t)r * I + cq);
                                sc[q][r] = e8m0_scale(__ldg(ws + (int64_t)r * mx.is + (cq >> 5)));
                            }
                        }
                    }
#pragma unroll
                    for (int q = 0; q < MX_UNR; ++q) {
                        const int cq = c + q * 512;
                        if (cq < I) {
#pragma unroll
                            for (int b = 0; b < DOWN_TB; ++b) {
                                if (b < nb) {
                                    const float *ar = act + (int64_t)arow[b] * I + cq;
                                    float af[16];
#pragma unroll
                                    for (int v = 0; v < 4; ++v) {
                                        const float4 a4 = ld_nc_f4(ar + 4 * v);
                                        af[4 * v] = a4.x;
                                        af[4 * v + 1] = a4.y;
                                        af[4 * v + 2] = a4.z;
                                        af[4 * v + 3] = a4.w;
                                    }
#pragma unroll
                                    for (int r = 0; r < DOWN_HW; ++r) {
                                        float wf[16];
                                        unpack16_e4m3(wv[q][r], wf);
                                        float p = 0.0f;
#pragma unroll
                                        for (int cc = 0; cc < 16; ++cc) p = fmaf(wf[cc], af[cc], p);
                                        acc[r][b] = fmaf(p, sc[q][r], acc[r][b]);
                                    }
                                }
                            }
                        }
                    }
                }
            } else {
            for (int c = lane * 8; c < I; c += 256 * DOWN_UNR) {
                uint4 wv[DOWN_UNR][DOWN_HW];
#pragma unroll
                for (int q = 0; q < DOWN_UNR; ++q) {
                    const int cq = c + q * 256;
                    if (cq < I) {
#pragma unroll
                        for (int r = 0; r < DOWN_HW; ++r) wv[q][r] = ld_stream16(wrow + (int64_t)r * I + cq);
                    }
                }
#pragma unroll
                for (int q = 0; q < DOWN_UNR; ++q) {
                    const int cq = c + q * 256;
                    if (cq < I) {
                        float wf[DOWN_HW][8];
#pragma unroll
                        for (int r = 0; r < DOWN_HW; ++r) unpack8(wv[q][r], wf[r]);
#pragma unroll
                        for (int b = 0; b < DOWN_TB; ++b) {
                            if (b < nb) {
                                const float *ar = act + (int64_t)arow[b] * I + cq;
                                const float4 v0 = ld_nc_f4(ar), v1 = ld_nc_f4(ar + 4);
                                const float af[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                                for (int r = 0; r < DOWN_HW; ++r)
#pragma unroll
                                    for (int cc = 0; cc < 8; ++cc) acc[r][b] = fmaf(wf[r][cc], af[cc], acc[r][b]);
                            }
                        }
                    }
                }
            }
            }
#pragma unroll
            for (int b = 0; b < DOWN_TB; ++b) {
                if (b < nb) {
#pragma unroll
                    for (int r = 0; r < DOWN_HW; ++r) {
                        const float v = warp_sum(acc[r][b]);
                        if (lane == 0) part[r * span + (arow[b] - a_lo)] = v;
                    }
                }
            }
        }
    }
    __syncthreads();
    // slot-ordered combine: out[t, h0+r] = sum_j w[t,j] * part[r][t,j]
    const int nt = t1 - t0;
    for (int q = threadIdx.x; q < DOWN_HW * nt; q += blockDim.x) {
        const int r = q / nt, tl = q - r * nt;
        const int t = t0 + tl;
        float o = 0.0f;
        for (int j = 0; j < k; ++j) o = fmaf(__ldg(wts + (int64_t)t * k + j), part[r * span + tl * k + j], o);
        out[(int64_t)t * H + h0 + r] = o;
    }
}

cudaError_t launch_decode_gate_up(const void *x, const void *wgu, const int32_t *uexp, const int32_t *ucount,
                                  const int32_t *offs, const int32_t *perm, int T, int H, int I, int E, int k,
                                  int warps, float *act, const FusedMx *mxw, cudaStream_t s)
{
    const int u_max = (int)((int64_t)T * k < E ? (int64_t)T * k : E);
    dim3 grid((unsigned)ceil_div(I, warps), (unsigned)u_max);
    DecodeMx mx{};
    if (mxw)
        mx = DecodeMx{(const uint8_t *)mxw->gq, (const uint8_t *)mxw->gs, (const uint8_t *)mxw->dq,
                      (const uint8_t *)mxw->ds, mx_scale_bytes(H), mx_scale_bytes(I)};
    auto kern = mxw ? (T == 1   ? decode_gate_up_kernel<1, true>
                       : T <= 2 ? decode_gate_up_kernel<2, true>
                       : T <= 4 ? decode_gate_up_kernel<4, true>
                                : decode_gate_up_kernel<8, true>)
                    : (T == 1   ? decode_gate_up_kernel<1, false>
                       : T <= 2 ? decode_gate_up_kernel<2, false>
                       : T <= 4 ? decode_gate_up_kernel<4, false>
                                : decode_gate_up_kernel<8, false>);
    kern<<<grid, warps * 32, 0, s>>>((const uint16_t *)x, (const uint16_t *)wgu, uexp, ucount, offs, perm, H, I, k,
                                     act, mx);
    return cudaPeekAtLastError();
}

cudaError_t decode_init_device()
{
    for (auto kern : {decode_down_kernel<1, false>, decode_down_kernel<2, false>, decode_down_kernel<4, false>,
                      decode_down_kernel<1, true>, decode_down_kernel<2, true>, decode_down_kernel<4, true>}) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int decode_down_tok_tile(int T, int k)
{
    // part[] is DOWN_HW * tok_tile * k floats; keep it at or under 64 KB.
    int tt = (64 * 1024) / (DOWN_HW * k * (int)sizeof(float));
    return T < tt ? T : tt;
}

cudaError_t launch_decode_down(const float *act, const void *wd, const float *w, const int32_t *uexp,
                               const int32_t *ucount, const int32_t *offs, const int32_t *perm, int T, int H,
                               int I, int k, int warps, float *out, const FusedMx *mxw, cudaStream_t s)
{
    const int tt = decode_down_tok_tile(T, k);
    dim3 grid((unsigned)(H / DOWN_HW), (unsigned)ceil_div(T, tt));
    const size_t smem = (size_t)DOWN_HW * tt * k * sizeof(float);
    DecodeMx mx{};
    if (mxw)
        mx = DecodeMx{(const uint8_t *)mxw->gq, (const uint8_t *)mxw->gs, (const uint8_t *)mxw->dq,
                      (const uint8_t *)mxw->ds, mx_scale_bytes(H), mx_scale_bytes(I)};
    auto kern = mxw ? (T == 1 ? decode_down_kernel<1, true> : T <= 2 ? decode_down_kernel<2, true>
                                                                     : decode_down_kernel<4, true>)
                    : (T == 1 ? decode_down_kernel<1, false> : T <= 2 ? decode_down_kernel<2, false>
                                                                      : decode_down_kernel<4, false>);
    kern<<<grid, warps * 32, smem, s>>>(act, (const uint16_t *)wd, w, uexp, ucount, offs, perm, T, H, I, k, tt,
                                        out, mx);
    return cudaPeekAtLastError();
}

}  // namespace moe
