"""The backward pass (moe_ffn_backward) against the FP64 backward oracle
(oracle/moe_backward.py) on the same bytes.

Acceptance per gradient (dx, dlogits, dW_gate_up, dW_down), as for the
forward output: ||g - g_ref||_2 / ||g_ref||_2 <= 1e-4 and max |g - g_ref| <=
1e-3 * rms(g_ref); an all-zero reference must be matched exactly (untouched
experts, one selected expert's logit gradient).  Shapes span ragged tiles
(I or H not a multiple of 128 or 256), experts with several 64-row chunks,
one expert, k = 32, skewed routing, tied and signed-zero logits, and the
training-size layer (sampled tokens and experts, the oracle fed only what
they need).  Plus: exact linearity in dout (2 dout gives twice every
gradient bit for bit, dout = 0 gives zeros), bit-identical
results across runs and launch widths, T = 0, a CUDA graph replay, a
workspace shared with the fused decode kernel's forward calls, and the
stage events."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth
from oracle import moe_backward as ob
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

NAMES = ("dx", "dlogits", "dwgu", "dwd")


@pytest.fixture(autouse=True)
def _no_faults():
    m.moe_ffn_device_faults(clear=True)
    yield
    assert m.moe_ffn_device_faults(clear=True) == 0, "a kernel's bounded wait gave up"


def _layer(wl, T, call=0, weights_device="cpu"):
    x, L, wgu, wd = gu.make_layer(wl, T, call=call, weights_device=weights_device)
    dout = synth.make_dout(wl, T, call=call, device="cuda")
    return x, L, wgu, wd, dout


def _gpu(x, L, wgu, wd, dout, k, **opt_fields):
    o = m.moe_ffn_opts()
    for f, v in opt_fields.items():
        setattr(o, f, v)
    got = m.moe_ffn_backward(x, L, wgu, wd, dout, k, opts=o)
    torch.cuda.synchronize()
    if x.shape[0]:
        assert o.path_taken == m.MOE_PATH_BACKWARD and o.n_stages == 11
    return dict(zip(NAMES, got))


def _oracle(x, L, wgu, wd, dout, k):
    return oracle.backward(synth.bf16_bits(x), L.cpu().numpy(), synth.bf16_bits(wgu), synth.bf16_bits(wd),
                           dout.cpu().numpy(), k)


def _accept(got, ref, what):
    g = got.detach().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    nw, mx, rms = gu.errors(g, ref)
    if rms == 0.0:
        assert mx == 0.0, f"{what}: reference is zero, result is not (max {mx:.3g})"
        return
    assert nw <= gu.NORMWISE_TOL, f"{what}: normwise {nw:.3g} > {gu.NORMWISE_TOL}"
    assert mx <= gu.MAXABS_RMS_TOL * rms, f"{what}: max abs {mx:.3g} > {gu.MAXABS_RMS_TOL}*rms ({rms:.3g})"


# (T, H, I, E, k, bias variance)
SMALL = [
    (4, 256, 128, 8, 2, 0.0),      # the tiny workload's shape
    (3, 64, 64, 4, 2, 0.0),        # one tile everywhere
    (37, 320, 192, 12, 3, 0.5),    # I = 192 and H = 320: partial 128-row and 256-column tiles
    (200, 128, 64, 4, 3, 0.0),     # 150 rows per expert: several chunks and K steps
    (64, 256, 128, 32, 1, 4.0),    # k = 1: the logit gradient is exactly zero; untouched experts
    (9, 128, 128, 1, 1, 0.0),      # one expert
    (50, 384, 256, 16, 8, 1.0),
    (17, 192, 320, 64, 32, 0.5),   # k = 32, many experts
    (64, 64, 64, 1024, 4, 1.0),    # 1024 experts: mostly one row each, 15 pad rows each, ~800 untouched
]


@pytest.mark.parametrize("T,H,I,E,k,bv", SMALL)
def test_backward_parity_small(T, H, I, E, k, bv):
    wl = gu.custom(T, H, I, E, k, bv, name="bwd_small")
    x, L, wgu, wd, dout = _layer(wl, T)
    got = _gpu(x, L, wgu, wd, dout, k)
    ref = _oracle(x, L, wgu, wd, dout, k)
    for n in NAMES:
        _accept(got[n], ref[n], f"{n} {T, H, I, E, k}")
    touched = set(ref["idx"].ravel().tolist())
    for e in set(range(E)) - touched:
        assert torch.count_nonzero(got["dwgu"][e]) == 0 and torch.count_nonzero(got["dwd"][e]) == 0
    if k == 1:
        assert torch.count_nonzero(got["dlogits"]) == 0


def test_backward_parity_mid_size():
    wl = gu.custom(256, 1024, 512, 32, 4, 0.5, name="bwd_mid")
    x, L, wgu, wd, dout = _layer(wl, 256, call=3)
    got = _gpu(x, L, wgu, wd, dout, 4)
    ref = _oracle(x, L, wgu, wd, dout, 4)
    for n in NAMES:
        _accept(got[n], ref[n], f"{n} mid")


def test_backward_is_exactly_linear_in_dout():
    """Every gradient is linear in dout, and every step of the path (the
    hi/lo splits, the MMAs' products and FP32 sums, the SwiGLU chain rule,
    the logit gradient) commutes with a power-of-two scale: 2 dout must give
    twice each gradient bit for bit, and dout = 0 exactly zero gradients."""
    wl = gu.custom(70, 320, 192, 12, 3, 1.0, name="bwd_linear")
    x, L, wgu, wd, dout = _layer(wl, 70, call=4)
    a = _gpu(x, L, wgu, wd, dout, 3)
    b = _gpu(x, L, wgu, wd, 2.0 * dout, 3)
    for n in NAMES:
        assert torch.equal(b[n], 2.0 * a[n]), n
    z = _gpu(x, L, wgu, wd, torch.zeros_like(dout), 3)
    for n in NAMES:
        assert torch.count_nonzero(z[n]) == 0, n


def test_backward_ties_and_signed_zero():
    """Logits drawn from {-1, -0.0, +0.0, 1}: the selection follows the
    lower-index rule on ties (-0.0 == +0.0), and the logit gradient lands on
    the experts the oracle selects."""
    T, H, I, E, k = 48, 256, 128, 16, 5
    wl = gu.custom(T, H, I, E, k, name="bwd_ties")
    x, _, wgu, wd, dout = _layer(wl, T, call=6)
    g = torch.Generator().manual_seed(11)
    vals = torch.tensor([-1.0, -0.0, 0.0, 1.0])
    L = vals[torch.randint(0, 4, (T, E), generator=g)].contiguous().cuda()
    got = _gpu(x, L, wgu, wd, dout, k)
    ref = _oracle(x, L, wgu, wd, dout, k)
    for n in NAMES:
        _accept(got[n], ref[n], f"{n} ties")
    mask = np.zeros((T, E), bool)
    mask[np.arange(T)[:, None], ref["idx"]] = True
    assert torch.count_nonzero(got["dlogits"].cpu()[torch.as_tensor(~mask)]) == 0


def test_backward_bit_identical_across_runs_and_widths():
    wl = gu.custom(96, 512, 256, 16, 4, 0.5, name="bwd_det")
    x, L, wgu, wd, dout = _layer(wl, 96, call=5)
    a = _gpu(x, L, wgu, wd, dout, 4)
    for opts in ({}, {"gemm_ctas": 37}, {"gemm_ctas": 1}):
        b = _gpu(x, L, wgu, wd, dout, 4, **opts)
        for n in NAMES:
            assert torch.equal(a[n], b[n]), (n, opts)


def test_backward_no_tokens_zeroes_weight_gradients():
    wl = gu.custom(0, 256, 128, 8, 2, name="bwd_t0")
    wgu, wd = synth.make_weights(wl, device="cuda")
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    L = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    dout = torch.empty((0, 256), dtype=torch.float32, device="cuda")
    dwgu = torch.full((8, 256, 256), float("nan"), device="cuda")
    dwd = torch.full((8, 256, 128), float("nan"), device="cuda")
    m.moe_ffn_backward(x, L, wgu, wd, dout, 2, dw_gate_up=dwgu, dw_down=dwd)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dwgu) == 0 and torch.count_nonzero(dwd) == 0


def test_backward_graph_replay_matches_eager():
    wl = gu.custom(40, 256, 128, 8, 2, 0.5, name="bwd_graph")
    x, L, wgu, wd, dout = _layer(wl, 40, call=2)
    ref = _gpu(x, L, wgu, wd, dout, 2)
    ws = m.new_backward_workspace(40, 256, 128, 8, 2)
    outs = [torch.full_like(ref[n], float("nan")) for n in NAMES]
    m.moe_ffn_backward(x, L, wgu, wd, dout, 2, *outs, workspace=ws)   # set-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        m.moe_ffn_backward(x, L, wgu, wd, dout, 2, *outs, workspace=ws, stream=s)
    for _ in range(2):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for n, o in zip(NAMES, outs):
            assert torch.equal(o, ref[n]), n


def test_backward_shares_a_workspace_with_fused_forward_calls():
    """Forward calls through the fused decode kernel keep state in their
    workspace; a backward call on the same bytes must leave that state
    consistent: every forward output equals a stateless call's bits, and the
    first fused call after a backward call meets at the grid barrier."""
    wl = synth.WORKLOADS["tiny_t4_h256_i128_e8_k2"]
    wgu, wd = synth.make_weights(wl, device="cuda")
    T, k = 4, wl.k
    ws = m.new_backward_workspace(T, wl.H, wl.I, wl.E, k)
    assert ws.numel() >= m.moe_ffn_workspace_bytes(T, wl.H, wl.I, wl.E, k)
    mode = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c in range(4):
        x, L = synth.make_tokens(wl, T, call=c, device="cuda")
        dout = synth.make_dout(wl, T, call=c, device="cuda")
        seen = []
        for _ in range(2):
            o = m.moe_ffn_opts()
            o.exchange_out = mode.data_ptr()
            out = m.moe_ffn_forward_ex(x, L, wgu, wd, k, workspace=ws, opts=o)
            torch.cuda.synchronize()
            assert o.path_taken == m.MOE_PATH_DECODE_FUSED
            seen.append(int(mode.item()))
            assert torch.equal(out, m.moe_ffn_forward(x, L, wgu, wd, k))
        assert seen == [m.EXCHANGE_BARRIER, m.EXCHANGE_TAGGED], seen
        got = m.moe_ffn_backward(x, L, wgu, wd, dout, k, workspace=ws)
        ref = m.moe_ffn_backward(x, L, wgu, wd, dout, k)
        torch.cuda.synchronize()
        for n, a, b in zip(NAMES, got, ref):
            assert torch.equal(a, b), n


def test_backward_stage_events():
    wl = gu.custom(64, 256, 128, 8, 2, name="bwd_stages")
    x, L, wgu, wd, dout = _layer(wl, 64)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_MAX_STAGES + 1)]
    for e in evs:
        e.record()
    arr = m.stage_event_array(evs)
    o = m.moe_ffn_opts()
    o.stage_events = m.ctypes.cast(arr, m.ctypes.c_void_p)
    m.moe_ffn_backward(x, L, wgu, wd, dout, 2, opts=o)
    torch.cuda.synchronize()
    assert o.n_stages == 11
    names = [m.moe_ffn_stage_name(m.MOE_PATH_BACKWARD, i) for i in range(o.n_stages)]
    assert names[0] == "router" and names[-1] == "dlogits"
    for i in range(o.n_stages):
        assert evs[i].elapsed_time(evs[i + 1]) >= 0.0


def test_backward_training_size_sampled():
    """The training-size layer (T = 2048, H = 6144, I = 2048, E = 256,
    k = 8, skewed routing): dx and dlogits of three tokens against the
    oracle on those tokens (handed only their experts), the weight
    gradients of three experts against the oracle's per-expert step on the
    rows routed to them, and a second run bit-identical to the first."""
    wl = synth.WORKLOADS["fwd_t2048_h6144_i2048_e256_k8_bias"]
    T, k = 2048, wl.k
    wgu, wd = synth.make_weights(wl, device="cuda")
    bias = synth.make_bias(wl)
    x, L = synth.make_tokens(wl, T, call=0, device="cuda", bias=bias)
    dout = synth.make_dout(wl, T, call=0, device="cuda")
    ws = m.new_backward_workspace(T, wl.H, wl.I, wl.E, k)
    got = m.moe_ffn_backward(x, L, wgu, wd, dout, k, workspace=ws)
    torch.cuda.synchronize()

    Ln = L.cpu().numpy()
    idx, w = oracle.route(Ln, k)
    # tokens: the oracle on their rows alone, with only their experts' weights
    toks = np.array([0, 1, T - 1])
    used = np.unique(idx[toks])
    emap = -np.ones(wl.E, np.int32)
    emap[used] = np.arange(len(used), dtype=np.int32)
    sel = torch.as_tensor(used, dtype=torch.long, device="cuda")
    tsel = torch.as_tensor(toks, dtype=torch.long, device="cuda")
    ref = oracle.backward(synth.bf16_bits(x[tsel]), Ln[toks], synth.bf16_bits(wgu.index_select(0, sel)),
                          synth.bf16_bits(wd.index_select(0, sel)), dout[tsel].cpu().numpy(), k, expert_map=emap)
    _accept(got[0][tsel], ref["dx"], "dx (sampled tokens)")
    _accept(got[1][tsel], ref["dlogits"], "dlogits (sampled tokens)")
    # experts: the per-expert step on every row routed to each
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    xf = ob.bf16_to_f64(synth.bf16_bits(x))
    df = dout.cpu().double().numpy()
    for e in sorted({0, int(np.argmax(counts)), wl.E - 1}):
        tok, slot = np.nonzero(idx == e)
        if len(tok) == 0:
            assert torch.count_nonzero(got[2][e]) == 0 and torch.count_nonzero(got[3][e]) == 0
            continue
        _, _, dwgu_e, dwd_e = ob.expert_backward(xf[tok], df[tok], w[tok, slot], synth.bf16_bits(wgu[e]),
                                                 synth.bf16_bits(wd[e]))
        _accept(got[2][e], dwgu_e, f"dW_gate_up expert {e} ({len(tok)} rows)")
        _accept(got[3][e], dwd_e, f"dW_down expert {e} ({len(tok)} rows)")
    again = m.moe_ffn_backward(x, L, wgu, wd, dout, k, workspace=ws)
    torch.cuda.synchronize()
    for n, a, b in zip(NAMES, got, again):
        assert torch.equal(a, b), n
