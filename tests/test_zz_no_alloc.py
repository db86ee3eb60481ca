"""moe_ffn_forward_noalloc: the forward pass for callers that cannot allocate
device memory once running (a latency-bound serving loop where an
allocation could synchronise the device or fail under memory pressure, or a
plugin whose host engine owns all device memory).  Its scratch is a fixed
device array inside the library, shared by all calls.

This file is collected last so that a run stopping at its first failure has
already run every other test; it passes alone in a fresh process too.
"""
import pytest
import torch

from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

# (T, H, I, E, k, bias variance, call): a fused decode call (tag region of
# 16 * 512 words in the shared array), and one whose routing and act rows
# land inside that region (T = 5: the grouped path)
SHAPE_A = (2, 1024, 512, 32, 4, 0.5, 0)
SHAPE_B = (5, 512, 256, 16, 2, 0.0, 1)


def _inputs(shape):
    T, H, I, E, k, bv, call = shape
    wl = gu.custom(T, H, I, E, k, bv, name=f"noalloc_{T}_{H}_{I}_{E}_{k}")
    x, L, wgu, wd = gu.make_layer(wl, T, call=call)
    return x, L, wgu, wd, k


def _noalloc(x, L, wgu, wd, k):
    out = torch.full((x.shape[0], x.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    return m.moe_ffn_forward_noalloc(x, L, wgu, wd, k, out=out)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    """Two consecutive calls with different inputs and shapes (so stale
    scratch from the first call would show in the second) give exactly the
    bits of moe_ffn_forward_ex with a workspace of its own -- the same
    kernels on the same inputs -- and meet the oracle's tolerance."""
    layers = [_inputs(s) for s in (SHAPE_A, SHAPE_B)]
    wants = [m.moe_ffn_forward_ex(*lay) for lay in layers]
    torch.cuda.synchronize()
    outs = [_noalloc(*lay) for lay in layers]     # the two calls, back to back
    torch.cuda.synchronize()
    for (x, L, wgu, wd, k), want, got in zip(layers, wants, outs):
        assert torch.equal(got, want)
        ref, ref_idx, ref_w = gu.oracle_ref(x, L, wgu, wd, k)
        nw, mx, rms = gu.errors(got.cpu(), ref)
        assert nw <= gu.NORMWISE_TOL, nw
        assert mx <= gu.MAXABS_RMS_TOL * rms, (mx, rms)
    assert m.moe_ffn_device_faults(clear=True) == 0


def test_noalloc_shape_a_b_a_a():
    """A fused call, a call of another shape whose regions fall inside the
    first one's tag region, then the first shape twice (the second of them
    exchanges act through tagged words in the shared array): each bit for bit
    equal to moe_ffn_forward_ex, and no bounded wait gives up."""
    a, b = _inputs(SHAPE_A), _inputs(SHAPE_B)
    want_a, want_b = m.moe_ffn_forward_ex(*a), m.moe_ffn_forward_ex(*b)
    torch.cuda.synchronize()
    for lay, want in ((a, want_a), (b, want_b), (a, want_a), (a, want_a)):
        got = _noalloc(*lay)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    assert m.moe_ffn_device_faults(clear=True) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    T, H, I, E, k = 4096, 6144, 2048, 8, 8   # workspace far above 16 MiB
    assert m.moe_ffn_workspace_bytes(T, H, I, E, k) > m.MOE_FFN_NOALLOC_SCRATCH_BYTES
    st = m.lib().moe_ffn_forward_noalloc(0x10000, 0x10000, 0x10000, 0x10000, T, H, I, E, k,
                                         0x10000, None)
    assert st == m.MOE_ERR_WORKSPACE_TOO_SMALL
