"""The training pair (moe_ffn_forward_train, then moe_ffn_backward_train):
the forward output against the oracle and, bit for bit, against the grouped
forward path; the gradients against the FP64 backward oracle and, bit for
bit, against moe_ffn_backward, which routes and recomputes gate/up itself.
The pair runs the same kernels in the same per-element order as those
entries, so any difference in a bit is a bug in what the state keeps.
Also: a second backward call on one state (another dout), a state no
forward call filled, T = 0, a CUDA graph of the whole training step, and
the training-size layer."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

NAMES = ("dx", "dlogits", "dwgu", "dwd")


@pytest.fixture(autouse=True)
def _no_faults():
    m.moe_ffn_device_faults(clear=True)
    yield
    assert m.moe_ffn_device_faults(clear=True) == 0, "a kernel's bounded wait gave up"


def _layer(wl, T, call=0):
    x, L, wgu, wd = gu.make_layer(wl, T, call=call)
    dout = synth.make_dout(wl, T, call=call, device="cuda")
    return x, L, wgu, wd, dout


def _grouped_forward(x, L, wgu, wd, k):
    o = m.moe_ffn_opts()
    o.path = m.MOE_PATH_GROUPED
    out = m.moe_ffn_forward_ex(x, L, wgu, wd, k, opts=o)
    torch.cuda.synchronize()
    return out


def _pair(x, L, wgu, wd, dout, k, state=None, **opt_fields):
    T, H = x.shape
    E, I = wgu.shape[0], wd.shape[2]
    if state is None:
        state = m.new_train_state(T, H, I, E, k)
    of, ob = m.moe_ffn_opts(), m.moe_ffn_opts()
    for o in (of, ob):
        for f, v in opt_fields.items():
            setattr(o, f, v)
    out = m.moe_ffn_forward_train(x, L, wgu, wd, k, state, opts=of)
    grads = m.moe_ffn_backward_train(x, L, wgu, wd, dout, k, state, opts=ob)
    torch.cuda.synchronize()
    if T:
        assert of.path_taken == m.MOE_PATH_TRAIN_FORWARD and of.n_stages == 5
        assert ob.path_taken == m.MOE_PATH_TRAIN_BACKWARD and ob.n_stages == 10
    return out, dict(zip(NAMES, grads)), state


SHAPES = [
    (4, 256, 128, 8, 2, 0.0),      # the tiny workload's shape
    (1, 256, 128, 8, 2, 0.0),      # one token
    (37, 320, 192, 12, 3, 0.5),    # partial tiles
    (200, 128, 64, 4, 3, 0.0),     # several 64-row chunks per expert
    (64, 256, 128, 32, 1, 4.0),    # k = 1, skewed routing, untouched experts
    (17, 192, 320, 64, 32, 0.5),   # k = 32
    (64, 64, 64, 1024, 4, 1.0),    # 1024 experts, most of them untouched
    (9, 128, 128, 1, 1, 0.0),      # one expert
]


@pytest.mark.parametrize("T,H,I,E,k,bv", SHAPES)
def test_train_pair_matches_the_separate_entries_and_the_oracle(T, H, I, E, k, bv):
    wl = gu.custom(T, H, I, E, k, bv, name="train_pair")
    x, L, wgu, wd, dout = _layer(wl, T, call=1)
    out, got, _ = _pair(x, L, wgu, wd, dout, k)
    assert torch.equal(out, _grouped_forward(x, L, wgu, wd, k))
    ref = m.moe_ffn_backward(x, L, wgu, wd, dout, k)
    torch.cuda.synchronize()
    for n, b in zip(NAMES, ref):
        assert torch.equal(got[n], b), n
    # and against the FP64 oracles on the same bytes
    fwd = oracle.forward(synth.bf16_bits(x), L.cpu().numpy(), synth.bf16_bits(wgu), synth.bf16_bits(wd), k)[0]
    nw, mx, rms = gu.errors(out.cpu().double().numpy(), fwd)
    assert nw <= gu.NORMWISE_TOL and mx <= gu.MAXABS_RMS_TOL * rms, (nw, mx, rms)
    bwd = oracle.backward(synth.bf16_bits(x), L.cpu().numpy(), synth.bf16_bits(wgu), synth.bf16_bits(wd),
                          dout.cpu().numpy(), k)
    for n in NAMES:
        nw, mx, rms = gu.errors(got[n].cpu().double().numpy(), bwd[n])
        if rms == 0.0:
            assert mx == 0.0, n
        else:
            assert nw <= gu.NORMWISE_TOL and mx <= gu.MAXABS_RMS_TOL * rms, (n, nw, mx, rms)


def test_backward_train_runs_again_on_one_state():
    """The backward call leaves the kept part of the state intact: a second
    call with another dout equals moe_ffn_backward with that dout."""
    wl = gu.custom(50, 384, 256, 16, 8, 1.0, name="train_again")
    x, L, wgu, wd, dout = _layer(wl, 50, call=2)
    _, first, state = _pair(x, L, wgu, wd, dout, 8)
    dout2 = synth.make_dout(wl, 50, call=7, device="cuda")
    again = m.moe_ffn_backward_train(x, L, wgu, wd, dout2, 8, state)
    ref2 = m.moe_ffn_backward(x, L, wgu, wd, dout2, 8)
    torch.cuda.synchronize()
    for n, a, b in zip(NAMES, again, ref2):
        assert torch.equal(a, b), n
    assert not torch.equal(again[0], first["dx"])


def test_backward_train_on_a_foreign_state_stays_in_bounds():
    """The backward call routes and sorts the logits itself and takes only
    the values g and u from the state: a state that no matching forward
    call filled (here every byte 0xFF, NaN as FP32) gives wrong gradients
    but no fault, and the same buffer then serves a proper pair."""
    wl = gu.custom(60, 256, 128, 16, 4, 1.0, name="train_foreign")
    x, L, wgu, wd, dout = _layer(wl, 60, call=5)
    state = m.new_train_state(60, 256, 128, 16, 4)
    state.fill_(255)
    bad = m.moe_ffn_backward_train(x, L, wgu, wd, dout, 4, state)
    torch.cuda.synchronize()
    assert torch.isnan(bad[0]).any()
    _, got, _ = _pair(x, L, wgu, wd, dout, 4, state=state)
    ref = m.moe_ffn_backward(x, L, wgu, wd, dout, 4)
    torch.cuda.synchronize()
    for n, b in zip(NAMES, ref):
        assert torch.equal(got[n], b), n


def test_train_pair_widths_and_no_tokens():
    wl = gu.custom(96, 512, 256, 16, 4, 0.5, name="train_widths")
    x, L, wgu, wd, dout = _layer(wl, 96, call=3)
    out, a, _ = _pair(x, L, wgu, wd, dout, 4)
    for ctas in (37, 1):
        out_c, b, _ = _pair(x, L, wgu, wd, dout, 4, gemm_ctas=ctas)
        assert torch.equal(out, out_c), ctas
        for n in NAMES:
            assert torch.equal(a[n], b[n]), (n, ctas)
    # T = 0: no output rows; the weight gradients are zeroed
    x0 = x[:0].contiguous()
    state = m.new_train_state(1, 512, 256, 16, 4)
    out0 = m.moe_ffn_forward_train(x0, L[:0].contiguous(), wgu, wd, 4, state)
    dwgu = torch.full_like(a["dwgu"], float("nan"))
    dwd = torch.full_like(a["dwd"], float("nan"))
    m.moe_ffn_backward_train(x0, L[:0].contiguous(), wgu, wd, dout[:0].contiguous(), 4, state, dw_gate_up=dwgu,
                             dw_down=dwd)
    torch.cuda.synchronize()
    assert out0.shape == (0, 512)
    assert torch.count_nonzero(dwgu) == 0 and torch.count_nonzero(dwd) == 0


def test_train_step_as_one_graph():
    """Forward and backward captured in one CUDA graph (a training step):
    replays equal the eager pair bit for bit."""
    wl = gu.custom(40, 256, 128, 8, 2, 0.5, name="train_graph")
    x, L, wgu, wd, dout = _layer(wl, 40, call=4)
    out_ref, ref, state = _pair(x, L, wgu, wd, dout, 2)
    out = torch.full_like(out_ref, float("nan"))
    grads = [torch.full_like(ref[n], float("nan")) for n in NAMES]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        m.moe_ffn_forward_train(x, L, wgu, wd, 2, state, out=out, stream=s)
        m.moe_ffn_backward_train(x, L, wgu, wd, dout, 2, state, *grads, stream=s)
    for _ in range(2):
        out.fill_(float("nan"))
        for g in grads:
            g.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_ref)
        for n, g in zip(NAMES, grads):
            assert torch.equal(g, ref[n]), n


def test_train_pair_training_size():
    """The training-size layer (T = 2048, H = 6144, I = 2048, E = 256,
    k = 8, skewed routing): the pair equals the grouped forward and
    moe_ffn_backward bit for bit (those two are checked against the oracles
    at this size elsewhere)."""
    wl = synth.WORKLOADS["fwd_t2048_h6144_i2048_e256_k8_bias"]
    T, k = 2048, wl.k
    wgu, wd = synth.make_weights(wl, device="cuda")
    x, L = synth.make_tokens(wl, T, call=0, device="cuda", bias=synth.make_bias(wl))
    dout = synth.make_dout(wl, T, call=0, device="cuda")
    out, got, state = _pair(x, L, wgu, wd, dout, k)
    del state
    assert torch.equal(out, _grouped_forward(x, L, wgu, wd, k))
    del out
    ref = m.moe_ffn_backward(x, L, wgu, wd, dout, k)
    torch.cuda.synchronize()
    for n, b in zip(NAMES, ref):
        assert torch.equal(got[n], b), n
    assert np.isfinite(got["dx"].sum().item())
