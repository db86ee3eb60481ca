"""Pins of the oracle's MXFP8 weight decoding (oracle/mxfp8.py) and of the
layer it feeds: the E4M3 and E8M0 tables against torch's own float8 types
(library conversions), the formats' closed-form values, the block structure
of the scales, and exact identities of the layer under scale changes."""
import numpy as np
import pytest
import torch

import oracle
from oracle import mxfp8 as mx


def _same(a, b):
    return np.array_equal(np.nan_to_num(a, nan=1234.5), np.nan_to_num(b, nan=1234.5))


def test_e4m3_table_matches_torch_float8():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert _same(mx.E4M3_TABLE, ref)


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0),
    (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x7E, 448.0), (0x81, -(2.0 ** -9)), (0xB8, -1.0),
    (0xFE, -448.0)])
def test_e4m3_closed_form(code, value):
    assert mx.e4m3_value(code) == value


def test_e4m3_signed_zero_and_nan():
    assert mx.e4m3_value(0x80) == 0.0 and np.signbit(mx.e4m3_value(0x80))
    assert np.isnan(mx.e4m3_value(0x7F)) and np.isnan(mx.e4m3_value(0xFF))
    finite = mx.E4M3_TABLE[np.isfinite(mx.E4M3_TABLE)]
    assert len(finite) == 254 and finite.max() == 448.0


def test_e8m0_table():
    assert mx.e8m0_value(127) == 1.0 and mx.e8m0_value(0) == 2.0 ** -127
    assert mx.e8m0_value(254) == 2.0 ** 127 and np.isnan(mx.e8m0_value(255))
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
        assert _same(mx.E8M0_TABLE, ref)


def test_scale_row_bytes():
    assert [mx.scale_row_bytes(K) for K in (32, 512, 768, 2048, 7168)] == [16, 16, 32, 64, 224]


def _codes(rng, shape):
    q = rng.integers(0, 256, size=shape, dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x30  # no NaN codes
    return q


def test_dequantize_block_structure():
    rng = np.random.default_rng(1)
    R, K = 3, 96
    q = _codes(rng, (R, K))
    s = np.full((R, mx.scale_row_bytes(K)), 127, np.uint8)
    s[:, K // 32:] = 255  # padding: ignored even where it holds the NaN scale
    base = mx.dequantize(q, s)
    assert np.array_equal(base, mx.E4M3_TABLE[q])
    s2 = s.copy()
    s2[1, 2] = 130  # block 2 of row 1: elements 64..95, times 8
    got = mx.dequantize(q, s2)
    want = base.copy()
    want[1, 64:96] *= 8.0
    assert np.array_equal(got, want)


def test_dequantize_rejects_nan_codes():
    q = np.zeros((1, 32), np.uint8)
    s = np.full((1, 16), 127, np.uint8)
    q[0, 5] = 0x7F
    with pytest.raises(ValueError):
        mx.dequantize(q, s)
    q[0, 5] = 0
    s[0, 0] = 255
    with pytest.raises(ValueError):
        mx.dequantize(q, s)


def test_bf16_conversion_is_exact_or_refuses():
    v = np.array([1.0, -448.0 * 2.0 ** 100, 2.0 ** -9 * 2.0 ** -120, 0.0])
    bits = mx.f64_to_bf16_exact(v)
    back = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(back, v)
    with pytest.raises(ValueError):
        mx.f64_to_bf16_exact(np.array([1.0 + 2.0 ** -10]))   # 11 significant bits
    with pytest.raises(ValueError):
        mx.f64_to_bf16_exact(np.array([2.0 ** -150]))        # below FP32's range


def _layer(rng, T=3, H=64, I=32, E=4, k=2):
    x = (rng.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    gq, dq = _codes(rng, (E, 2 * I, H)), _codes(rng, (E, H, I))
    gs = rng.integers(120, 125, size=(E, 2 * I, mx.scale_row_bytes(H)), dtype=np.uint8)
    ds = rng.integers(120, 125, size=(E, H, mx.scale_row_bytes(I)), dtype=np.uint8)
    return x, logits, gq, gs, dq, ds, k


def test_forward_mxfp8_unit_scales_equals_bf16_layer():
    # scale 127 everywhere: the weights are the E4M3 values themselves, which
    # the BF16 layer can take directly
    rng = np.random.default_rng(2)
    x, logits, gq, gs, dq, ds, k = _layer(rng)
    gs[:] = 127
    ds[:] = 127
    got = oracle.forward_mxfp8(x, logits, gq, gs, dq, ds, k)[0]
    wgu = mx.f64_to_bf16_exact(mx.E4M3_TABLE[gq])
    wd = mx.f64_to_bf16_exact(mx.E4M3_TABLE[dq])
    assert np.array_equal(got, oracle.forward(x, logits, wgu, wd, k)[0])


def test_forward_mxfp8_down_scales_double_the_output():
    rng = np.random.default_rng(3)
    x, logits, gq, gs, dq, ds, k = _layer(rng)
    out = oracle.forward_mxfp8(x, logits, gq, gs, dq, ds, k)[0]
    out2 = oracle.forward_mxfp8(x, logits, gq, gs, dq, ds + 1, k)[0]
    assert np.array_equal(out2, 2.0 * out)


def test_forward_mxfp8_up_scales_double_the_output():
    # act = silu(gate) * up: doubling the up rows (2I rows: gate i, then up
    # I + i) doubles every act value and so the output; doubling the gate
    # rows does not
    rng = np.random.default_rng(4)
    x, logits, gq, gs, dq, ds, k = _layer(rng)
    I = gq.shape[1] // 2
    out = oracle.forward_mxfp8(x, logits, gq, gs, dq, ds, k)[0]
    up = gs.copy()
    up[:, I:] += 1
    assert np.array_equal(oracle.forward_mxfp8(x, logits, gq, up, dq, ds, k)[0], 2.0 * out)
    gate = gs.copy()
    gate[:, :I] += 1
    assert not np.array_equal(oracle.forward_mxfp8(x, logits, gq, gate, dq, ds, k)[0], 2.0 * out)
