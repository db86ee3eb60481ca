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


def _check_close(got, want):
    nw, mx, rms = gu.errors(got.cpu(), want.cpu().double().numpy())
    assert nw <= gu.NORMWISE_TOL, nw
    assert mx <= gu.MAXABS_RMS_TOL * rms, (mx, rms)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    """Two consecutive calls with different inputs and shapes (so stale
    scratch from the first call would show in the second) agree with
    moe_ffn_forward_ex within the parity tolerance."""
    cases = [(2, 1024, 512, 32, 4, 0.5, 0), (5, 512, 256, 16, 2, 0.0, 1)]
    layers = []
    for T, H, I, E, k, bv, call in cases:
        wl = gu.custom(T, H, I, E, k, bv, name=f"noalloc_{T}_{H}_{I}_{E}_{k}")
        x, L, wgu, wd = gu.make_layer(wl, T, call=call)
        want = m.moe_ffn_forward_ex(x, L, wgu, wd, k)
        layers.append((x, L, wgu, wd, k, want))
    torch.cuda.synchronize()
    outs = []
    for x, L, wgu, wd, k, _ in layers:     # the two calls, back to back
        out = torch.empty((x.shape[0], x.shape[1]), dtype=torch.float32, device="cuda")
        outs.append(m.moe_ffn_forward_noalloc(x, L, wgu, wd, k, out=out))
    torch.cuda.synchronize()
    for (_, _, _, _, _, want), got in zip(layers, outs):
        _check_close(got, want)
    assert m.moe_ffn_device_faults(clear=True) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    T, H, I, E, k = 4096, 6144, 2048, 8, 8   # workspace far above 16 MiB
    assert m.moe_ffn_workspace_bytes(T, H, I, E, k) > m.MOE_FFN_NOALLOC_SCRATCH_BYTES
    st = m.lib().moe_ffn_forward_noalloc(0x10000, 0x10000, 0x10000, 0x10000, T, H, I, E, k,
                                         0x10000, None)
    assert st == m.MOE_ERR_WORKSPACE_TOO_SMALL
