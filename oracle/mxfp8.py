"""MXFP8 expert weights for the oracle: decoding and exact dequantisation.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): the product never
imports it and it imports nothing of the product.

What it computes.  The Mixture-of-Kittens article ("커서가 MoE 학습 메가커널
믹스처 오브 키튼스를 아파치 2.0으로 공개했다", section 2.37배는 어떤 기준선과
비교한 숫자인가) measures the MoE layer with MXFP8 operands; the pages do not
write the format out.  The layer's reading is the MX format as the OCP
Microscaling Formats (MX) v1.0 specification defines MXFP8, applied to the
expert weights only (the activations stay BF16):

  * every row of W_gate_up [E, 2I, H] and W_down [E, H, I] is cut into
    blocks of 32 consecutive elements along the reduction axis (H for
    W_gate_up, I for W_down);
  * each element is an FP8 E4M3 code (OCP 8-bit floating point, "OFP8"):
    sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 holds
    the subnormals m/8 * 2^-6; the code S.1111.111 is NaN; there is no
    infinity, so the largest magnitude is 1.75 * 2^8 = 448;
  * each block has one E8M0 scale: an unsigned 8-bit exponent, value
    2^(s - 127); s = 255 is NaN;
  * the weight is the element's value times its block's scale.

The layer is then the BF16 layer's definition (``moe_oracle.c``) applied to
these weights.  An E4M3 value has 4 significant bits, so every weight is a
BF16 number (8 significant bits) whenever its exponent lies in BF16's range;
``dequantize_bf16`` converts exactly and refuses anything else, and the
FP64 oracle then runs on exactly the weights the format denotes.

Memory layout of the scales (the spec leaves it to the implementation): for
a matrix with rows of K elements the scales are [rows, Ks] bytes with
Ks = ceil(K / 32) rounded up to a multiple of 16; bytes past K / 32 in a row
are padding and ignored.  K must be a multiple of 32.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32


def scale_row_bytes(K: int) -> int:
    """Bytes per row of the scale array for rows of K elements."""
    assert K % BLOCK == 0
    return -(-(K // BLOCK) // 16) * 16


def e4m3_value(code: int) -> float:
    """The value of one E4M3 code (0..255), from the format's definition;
    NaN for the two NaN codes."""
    code = int(code)
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# the 256 values as a lookup table (float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e8m0_value(code: int) -> float:
    """The value 2^(code - 127) of one E8M0 scale; NaN for 255."""
    code = int(code)
    if code == 255:
        return float("nan")
    return 2.0 ** (code - 127)


E8M0_TABLE = np.array([e8m0_value(c) for c in range(256)], dtype=np.float64)


def dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Weights in float64 from E4M3 codes q [..., K] (uint8) and E8M0 scales
    s [..., Ks] (uint8, Ks = scale_row_bytes(K)): element j of a row times
    the scale of block j // 32 of that row.  Raises on NaN codes."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    K = q.shape[-1]
    nb = K // BLOCK
    assert K % BLOCK == 0 and s.shape[:-1] == q.shape[:-1] and s.shape[-1] == scale_row_bytes(K)
    vals = E4M3_TABLE[q]
    scales = E8M0_TABLE[s[..., :nb]]
    if np.isnan(vals).any() or np.isnan(scales).any():
        raise ValueError("MXFP8 weights hold a NaN code")
    return vals * np.repeat(scales, BLOCK, axis=-1)


def f64_to_bf16_exact(v: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) of float64 values that BF16 represents
    exactly; raises if any does not."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    f = v.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), v):
        raise ValueError("a weight is outside FP32's exact range")
    bits = f.view(np.uint32)
    if (bits & 0xFFFF).any():
        raise ValueError("a weight is not a BF16 number")
    return (bits >> 16).astype(np.uint16)


def dequantize_bf16(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The dequantised weights as exact BF16 bit patterns (uint16)."""
    return f64_to_bf16_exact(dequantize(q, s))
