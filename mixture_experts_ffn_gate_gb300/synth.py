"""Seeded synthetic inputs for the routed MoE SwiGLU FFN layer.

This module holds the workload table and the random-input recipe, and nothing
of the layer's arithmetic: it is the one module that both the CUDA path's
callers and the FP64 oracle's callers use.

Recipe (every tensor is drawn in FP32 and rounded to BF16 round-to-nearest-even
with ``Tensor.to(torch.bfloat16)``):

* ``x``           [T, H]      ~ N(0, 1)                         -> BF16
* ``logits``      [T, E]      ~ N(0, 1) + bias[e]                  (FP32)
* ``bias``        [E]         ~ N(0, var) drawn once per workload (var 0 = none)
* ``w_gate_up``   [E, 2I, H]  ~ N(0, 1/H) (fan-in H)            -> BF16
* ``w_down``      [E, H, I]   ~ N(0, 1/I) (fan-in I)            -> BF16
* ``w_router``    [E, H]      ~ N(0, 1/H) (fan-in H)            -> BF16
  (calls that pass the router weights; their logits are x . W_r^T + bias)
* ``dout``        [T, H]      ~ N(0, 1)                            (FP32)
  (the upstream gradient of the backward pass)

``N(0, v)`` names the variance, so std = sqrt(v).  Each expert's weights come
from a generator seeded with ``seed_for(workload, tensor, expert)``; token
batches are seeded per call index, so "fresh tokens" for call n are always the
same bytes.  Large weight sets are drawn on the GPU (one expert at a time, so
the FP32 temporary stays small); whoever needs them on the host reads back the
exact BF16 bytes.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: tuple          # token counts this workload is run at
    H: int
    I: int
    E: int
    k: int
    bias_var: float   # variance of the per-expert logit bias (0 = no bias)
    about: str

    def weight_bytes(self) -> int:
        return self.E * 3 * self.H * self.I * 2


# The five layer shapes.  Names say what each one is and its sizes.
WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_t4_h256_i128_e8_k2", (4,), 256, 128, 8, 2, 0.0,
                 "tiny layer for full oracle comparison"),
        Workload("decode_h2048_i768_e128_k8", (1, 2), 2048, 768, 128, 8, 0.0,
                 "Qwen-3-style decode layer"),
        Workload("decode_h4096_i1536_e128_k8_bias", (1, 4, 16, 64), 4096, 1536,
                 128, 8, 0.5, "larger Qwen-3-style decode sweep, skewed routing"),
        Workload("decode_h7168_i2048_e384_k8_bias", (1, 8, 32), 7168, 2048, 384,
                 8, 0.5, "wide-expert decode (384 experts, hidden 7168)"),
        Workload("fwd_t2048_h6144_i2048_e256_k8_bias", (2048,), 6144, 2048, 256,
                 8, 1.0, "training-size forward, skewed expert loads"),
    ]
}


def seed_for(*parts) -> int:
    """A stable 63-bit seed from any tuple of names and numbers."""
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, std, device, seed):
    t = torch.randn(shape, generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def make_weights(wl: Workload, device="cpu", *, H=None, I=None, E=None, experts=None, layer=0):
    """Expert weights (w_gate_up [E,2I,H], w_down [E,H,I]) as BF16 on device.

    H, I, E default to the workload's; tests pass smaller ones to reuse the
    recipe at other sizes.  ``experts`` (a list of expert ids) draws only
    those blocks, in that order, with the same seeds as the full set.
    ``layer`` > 0 draws another layer's weights (same distribution, other
    seeds), for running calls over several layers.
    """
    tag = () if layer == 0 else ("layer", layer)
    H = H or wl.H
    I = I or wl.I
    E = E or wl.E
    ids = list(range(E)) if experts is None else list(experts)
    wgu = torch.empty((len(ids), 2 * I, H), dtype=torch.bfloat16, device=device)
    wd = torch.empty((len(ids), H, I), dtype=torch.bfloat16, device=device)
    for j, e in enumerate(ids):
        wgu[j] = _randn((2 * I, H), 1.0 / math.sqrt(H), device,
                        seed_for(wl.name, H, I, "w_gate_up", e, *tag)).to(torch.bfloat16)
        wd[j] = _randn((H, I), 1.0 / math.sqrt(I), device,
                       seed_for(wl.name, H, I, "w_down", e, *tag)).to(torch.bfloat16)
    return wgu, wd


MX_BLOCK = 32  # MXFP8: elements per E8M0 scale, along the reduction axis


def mx_scale_row_bytes(K: int) -> int:
    """Bytes per row of an MXFP8 scale array for rows of K elements:
    K / 32 scales, padded to a multiple of 16 bytes."""
    return -(-(K // MX_BLOCK) // 16) * 16


def _quantize_mx(w: torch.Tensor):
    """Rows of float32 weights [R, K] -> (E4M3 codes uint8 [R, K], E8M0
    scales uint8 [R, Ks]): per block of 32, the scale 2^(floor(log2 amax) -
    8) (amax maps into [256, 512), as the MX specification's conversion
    recipe does for E4M3, whose largest exponent is 8), then each element
    divided by it (exact) and rounded to E4M3 (nearest, ties to even),
    clamped to +-448.  Input generation only: the recipe that turns the
    seeded Gaussian weights into MXFP8 ones."""
    R, K = w.shape
    b = w.view(R, K // MX_BLOCK, MX_BLOCK)
    amax = b.abs().amax(-1)
    e = torch.frexp(amax).exponent.to(torch.int32) - 1  # floor(log2 amax) for amax > 0
    sc = torch.where(amax > 0, e - 8 + 127, torch.full_like(e, 127)).clamp(1, 254)
    x = torch.ldexp(b, (127 - sc).to(torch.float32).unsqueeze(-1))
    q = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).view(R, K)
    s_full = torch.zeros((R, mx_scale_row_bytes(K)), dtype=torch.uint8, device=w.device)
    s_full[:, : K // MX_BLOCK] = sc.to(torch.uint8)
    return q, s_full


def make_weights_mxfp8(wl: Workload, device="cpu", *, H=None, I=None, E=None, experts=None, layer=0):
    """MXFP8 expert weights: (wgu_q uint8 [E, 2I, H], wgu_s uint8 [E, 2I,
    Hs], wd_q uint8 [E, H, I], wd_s uint8 [E, H, Is]) -- the same seeded
    Gaussian draws as make_weights (N(0, 1/H) and N(0, 1/I)), quantised by
    _quantize_mx instead of rounded to BF16.  Arguments as for
    make_weights."""
    tag = () if layer == 0 else ("layer", layer)
    H = H or wl.H
    I = I or wl.I
    E = E or wl.E
    ids = list(range(E)) if experts is None else list(experts)
    n = len(ids)
    gq = torch.empty((n, 2 * I, H), dtype=torch.uint8, device=device)
    gs = torch.empty((n, 2 * I, mx_scale_row_bytes(H)), dtype=torch.uint8, device=device)
    dq = torch.empty((n, H, I), dtype=torch.uint8, device=device)
    ds = torch.empty((n, H, mx_scale_row_bytes(I)), dtype=torch.uint8, device=device)
    for j, e in enumerate(ids):
        gq[j], gs[j] = _quantize_mx(_randn((2 * I, H), 1.0 / math.sqrt(H), device,
                                           seed_for(wl.name, H, I, "w_gate_up", e, *tag)))
        dq[j], ds[j] = _quantize_mx(_randn((H, I), 1.0 / math.sqrt(I), device,
                                           seed_for(wl.name, H, I, "w_down", e, *tag)))
    return gq, gs, dq, ds


def make_router(wl: Workload, device="cpu", *, H=None, E=None, layer=0):
    """Router weights W_r [E, H] ~ N(0, 1/H) -> BF16 (a linear layer's
    weight, one row per expert), for calls that pass the router weights
    instead of logits; the per-expert bias of such calls is make_bias."""
    tag = () if layer == 0 else ("layer", layer)
    H = H or wl.H
    E = E or wl.E
    return _randn((E, H), 1.0 / math.sqrt(H), device, seed_for(wl.name, H, E, "w_router", *tag)).to(torch.bfloat16)


def make_bias(wl: Workload, E=None, device="cpu"):
    E = E or wl.E
    if wl.bias_var == 0.0:
        return torch.zeros(E, dtype=torch.float32, device=device)
    return _randn((E,), math.sqrt(wl.bias_var), "cpu",
                  seed_for(wl.name, E, "bias")).to(device)


def make_tokens(wl: Workload, T: int, call: int = 0, device="cpu", *, H=None,
                E=None, bias=None):
    """Token activations x [T,H] BF16 and router logits [T,E] FP32 for call n."""
    H = H or wl.H
    E = E or wl.E
    x = _randn((T, H), 1.0, "cpu", seed_for(wl.name, H, "x", T, call))
    logits = _randn((T, E), 1.0, "cpu", seed_for(wl.name, E, "logits", T, call))
    if bias is None:
        bias = make_bias(wl, E)
    logits += bias.to("cpu")[None, :]
    return x.to(torch.bfloat16).to(device), logits.to(device)


def make_dout(wl: Workload, T: int, call: int = 0, device="cpu", *, H=None):
    """The upstream gradient dL/dout [T,H] FP32 ~ N(0, 1) for call n."""
    H = H or wl.H
    return _randn((T, H), 1.0, "cpu", seed_for(wl.name, H, "dout", T, call)).to(device)


def bf16_bits(t: torch.Tensor):
    """Raw 16-bit patterns of a BF16 tensor as a numpy uint16 array (host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
