"""FP64-exact router projection for the oracle: the step before top-k.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): the product never
imports it and it imports nothing of the product.

What it computes.  The warp-decode article ("Cursor warp decode 공개 ...",
section 배경 및 맥락) names expert routing as the step that picks each token's
experts; neither page writes the router out.  The layer's reading: a linear
map of the token's activation to one score per expert plus a per-expert
bias,

    logits[t, e] = round_f32( sum_h x[t, h] * W_r[e, h] + b[e] ),

with x and W_r in BF16 (W_r laid out [E, H], one row per expert, as a linear
layer's weight), b in FP32, the sum taken exactly and rounded once to FP32
(round to nearest, ties to even).  Rounding once from the exact value makes
the logits a function of the inputs alone, so the top-k selection that
follows (an integer decision) is the same wherever it is computed.

How.  Each product of two BF16 values is exact in FP64 (8 + 8 significant
bits), so the exact sum of the products and the bias is the exact sum of FP64
numbers; ``math.fsum`` returns it rounded once to FP64.  Rounding that FP64
value to FP32 gives the FP32 rounding of the exact sum except when the FP64
value sits exactly halfway between two FP32 neighbours (double rounding):
then the exact sum is formed with ``fractions.Fraction`` and rounded
directly.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> their exact values as float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_f32_exact(terms) -> np.float32:
    """The exact sum of the float64 ``terms``, rounded once to float32."""
    s = math.fsum(terms)
    f = np.float32(s)
    if not math.isfinite(s) or float(f) == s:
        return f
    # neighbours of s in float32; s halfway between them is the one case where
    # rounding s again can differ from rounding the exact sum
    lo, hi = (f, np.nextafter(f, np.float32(np.inf))) if float(f) < s else (np.nextafter(f, np.float32(-np.inf)), f)
    mid = (Fraction(float(lo)) + Fraction(float(hi))) / 2
    if Fraction(s) != mid:
        return f
    exact = sum((Fraction(float(v)) for v in terms), Fraction(0))
    if exact > mid:
        return hi
    if exact < mid:
        return lo
    return lo if (int(lo.view(np.uint32)) & 1) == 0 else hi


def router_logits(x_bits: np.ndarray, wr_bits: np.ndarray, bias=None) -> np.ndarray:
    """logits float32 [T, E] from x bf16 bits [T, H], W_r bf16 bits [E, H]
    and an optional float32 bias [E]; see the module docstring."""
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(wr_bits)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape == (E, H)
    b = np.zeros(E, np.float64) if bias is None else np.asarray(bias, np.float32).astype(np.float64)
    assert b.shape == (E,)
    out = np.empty((T, E), np.float32)
    for t in range(T):
        for e in range(E):
            prods = x[t] * w[e]          # exact: products of BF16 values fit FP64
            out[t, e] = round_f32_exact([*prods.tolist(), float(b[e])])
    return out
