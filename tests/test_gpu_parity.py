"""GPU parity: the CUDA path through the C ABI against the FP64 oracle on the
same seeded bytes, element by element, on sizes the oracle finishes in
seconds (several tiles and a ragged tail), on edge cases, and on metamorphic
properties that must hold bit-exactly."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PATH_IDS = ["decode", "grouped"]


@pytest.fixture(autouse=True)
def _no_faults():
    yield
    assert m.moe_ffn_device_faults(clear=True) == 0, "a kernel's bounded wait gave up"


@pytest.mark.parametrize("path", PATH_IDS)
def test_tiny_workload(path):
    wl = synth.WORKLOADS["tiny_t4_h256_i128_e8_k2"]
    x, L, wgu, wd = gu.make_layer(wl, 4)
    out, idx, w = gu.run_gpu(x, L, wgu, wd, wl.k, path)
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, L, wgu, wd, wl.k), what=wl.name)


# (T, H, I, E, k, bias_var): several tiles, ragged tails (H or I not a
# multiple of 128/256), k = 1, k = E, a single expert, skewed routing.
SHAPES = [
    (1, 256, 128, 8, 2, 0.0),
    (3, 320, 192, 5, 3, 0.0),
    (37, 512, 192, 16, 4, 0.5),
    (64, 384, 320, 12, 1, 0.0),
    (9, 256, 128, 6, 6, 0.0),
    (5, 128, 64, 1, 1, 0.0),
    (130, 640, 256, 32, 8, 1.0),
    (300, 256, 128, 4, 2, 4.0),   # heavy skew: > 256 tokens on one expert
]


@pytest.mark.parametrize("path", PATH_IDS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "T%d_H%d_I%d_E%d_k%d" % s[:5])
def test_shapes(path, shape):
    T, H, I, E, k, bv = shape
    wl = gu.custom(T, H, I, E, k, bv, name="shape_%d_%d_%d_%d_%d" % shape[:5])
    x, L, wgu, wd = gu.make_layer(wl, T)
    out, idx, w = gu.run_gpu(x, L, wgu, wd, k, path)
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, L, wgu, wd, k), what=str(shape))


@pytest.mark.parametrize("path", PATH_IDS)
def test_exact_ties_and_signed_zero(path):
    """Logits drawn from {-1, 0, 1} (and -0.0): ties everywhere; indices must
    match the oracle's lower-index rule bit for bit."""
    T, H, I, E, k = 40, 256, 128, 16, 5
    wl = gu.custom(T, H, I, E, k, name="ties")
    x, _, wgu, wd = gu.make_layer(wl, T)
    g = torch.Generator().manual_seed(5)
    L = (torch.randint(-1, 2, (T, E), generator=g).float())
    L[L == 0] = -0.0 * torch.ones_like(L[L == 0])
    L[::2, 3] = 0.0
    L = L.cuda()
    out, idx, w = gu.run_gpu(x, L, wgu, wd, k, path)
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, L, wgu, wd, k), what="ties")


def _tie_logits(T, E, seed):
    """Logits drawn from {-1, -0.0, +0.0, 1}: ties everywhere, and signed
    zeros that must compare equal."""
    g = torch.Generator().manual_seed(seed)
    vals = torch.tensor([-1.0, -0.0, 0.0, 1.0])
    return vals[torch.randint(0, 4, (T, E), generator=g)].contiguous()


def _fused_and_general_agree(x, L, wgu, wd, k):
    """The tokens (T <= 4) through the fused decode kernel, checked against
    the oracle, and bit for bit against the same tokens inside a batch of
    eight, which the general decode kernels (router kernel included) take."""
    T, H = x.shape
    E = L.shape[1]
    o = m.moe_ffn_opts()
    o.path = m.MOE_PATH_DECODE
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = m.moe_ffn_forward_ex(x, L, wgu, wd, k, topk_idx=idx, topk_w=w, opts=o)
    torch.cuda.synchronize()
    assert o.path_taken == m.MOE_PATH_DECODE_FUSED
    out, idx, w = out.cpu(), idx.cpu(), w.cpu()
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, L, wgu, wd, k), what=f"fused T={T} k={k}")
    x8 = torch.cat([x, x[:1].expand(8 - T, H)]).contiguous()
    L8 = torch.cat([L, L[:1].expand(8 - T, E)]).contiguous()
    out8, idx8, w8 = gu.run_gpu(x8, L8, wgu, wd, k, "decode")
    assert torch.equal(idx8[:T], idx)
    assert torch.equal(w8[:T], w)
    assert torch.equal(out8[:T], out)


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_ties_and_signed_zero_through_the_fused_kernel(T):
    """The tie rule (lower index wins, -0.0 == +0.0) where the headline
    decode calls route: inside the fused decode kernel."""
    H, I, E, k = 256, 128, 16, 5
    wl = gu.custom(T, H, I, E, k, name="fused_ties")
    x, _, wgu, wd = gu.make_layer(wl, T)
    L = _tie_logits(T, E, seed=10 + T)
    L[0, 3] = -0.0          # a signed zero on a likely winner's tie
    L[0, 2] = 0.0
    _fused_and_general_agree(x, L.cuda(), wgu, wd, k)


@pytest.mark.parametrize("T,E,k", [(1, 300, 8), (3, 1024, 8), (4, 1024, 7), (2, 130, 1)])
def test_fused_routing_ties_many_experts(T, E, k):
    """The fused kernel's routing (k <= 8: each lane's keys through the
    sorting network, 8 at a time, then merged) on ties and signed zeros, with
    E up to 1024 and ragged: the same bits as the router kernel of the
    general decode path, and the oracle's indices."""
    H, I = 256, 128
    wl = gu.custom(T, H, I, E, k, name="fused_routing_ties")
    x, _, wgu, wd = gu.make_layer(wl, T)
    L = _tie_logits(T, E, seed=40 + T + E)
    _fused_and_general_agree(x, L.cuda(), wgu, wd, k)


@pytest.mark.parametrize("T,k", [(4, 9), (4, 16), (1, 32), (2, 32)])
def test_ties_in_the_rescan_branch(T, k):
    """k > 8 selects by rescanning the lane's keys below the last winner
    (the register list holds eight); with tied logits the keys still order
    by index.  Through the fused kernel and the router kernel."""
    H, I, E = 128, 64, 64
    wl = gu.custom(T, H, I, E, k, name="rescan_ties")
    x, _, wgu, wd = gu.make_layer(wl, T)
    L = _tie_logits(T, E, seed=100 + k + T).cuda()
    _fused_and_general_agree(x, L, wgu, wd, k)


@pytest.mark.parametrize("path", PATH_IDS)
@pytest.mark.parametrize("k", [9, 16, 32])
def test_ties_in_the_rescan_branch_many_tokens(path, k):
    """The router kernel's rescan branch over 40 tokens of tied logits."""
    T, H, I, E = 40, 128, 64, 64
    wl = gu.custom(T, H, I, E, k, name="rescan_ties_many")
    x, _, wgu, wd = gu.make_layer(wl, T)
    L = _tie_logits(T, E, seed=200 + k).cuda()
    out, idx, w = gu.run_gpu(x, L, wgu, wd, k, path)
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, L, wgu, wd, k), what=f"rescan k={k}")


@pytest.mark.parametrize("path", PATH_IDS)
def test_zero_input_gives_zero(path):
    T, H, I, E, k = 7, 256, 128, 8, 2
    wl = gu.custom(T, H, I, E, k, name="zero")
    x, L, wgu, wd = gu.make_layer(wl, T)
    out, _, _ = gu.run_gpu(torch.zeros_like(x), L, wgu, wd, k, path)
    assert torch.all(out == 0)


def test_zero_tokens():
    wl = synth.WORKLOADS["tiny_t4_h256_i128_e8_k2"]
    _, _, wgu, wd = gu.make_layer(wl, 4)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    L = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    out = m.moe_ffn_forward(x, L, wgu, wd, 2)
    assert out.shape == (0, 256)
    out = m.moe_ffn_forward_ex(x, L, wgu, wd, 2)
    assert out.shape == (0, 256)


@pytest.mark.parametrize("path", PATH_IDS)
def test_metamorphic_bit_exact(path):
    """Token permutation permutes rows; a token alone equals the same token
    inside the batch; doubling W_down doubles the output -- all bit for bit."""
    T, H, I, E, k = 24, 512, 256, 16, 4
    wl = gu.custom(T, H, I, E, k, 0.5, name="meta")
    x, L, wgu, wd = gu.make_layer(wl, T)
    out, _, _ = gu.run_gpu(x, L, wgu, wd, k, path)
    p = torch.randperm(T, generator=torch.Generator().manual_seed(3))
    outp, _, _ = gu.run_gpu(x[p.cuda()].contiguous(), L[p.cuda()].contiguous(), wgu, wd, k, path)
    assert torch.equal(outp, out[p])
    for t in (0, 11, T - 1):
        o1, _, _ = gu.run_gpu(x[t:t + 1].contiguous(), L[t:t + 1].contiguous(), wgu, wd, k, path)
        assert torch.equal(o1[0], out[t]), t
    out2, _, _ = gu.run_gpu(x, L, wgu, (wd.float() * 2).to(torch.bfloat16), k, path)
    assert torch.equal(out2, out * 2)


@pytest.mark.parametrize("path", PATH_IDS)
def test_repeatable_100_runs(path):
    T, H, I, E, k = 48, 512, 256, 32, 8
    wl = gu.custom(T, H, I, E, k, 1.0, name="repeat")
    x, L, wgu, wd = gu.make_layer(wl, T)
    first, idx0, w0 = gu.run_gpu(x, L, wgu, wd, k, path)
    ws = m.new_workspace(T, H, I, E, k)
    o = m.moe_ffn_opts()
    o.path = gu.PATHS[path]
    outs = [m.moe_ffn_forward_ex(x, L, wgu, wd, k, workspace=ws, opts=o) for _ in range(100)]
    torch.cuda.synchronize()
    for r in outs:
        assert torch.equal(r.cpu(), first)


def test_decode_launch_config_sweep():
    T, H, I, E, k = 20, 768, 320, 24, 6
    wl = gu.custom(T, H, I, E, k, 0.5, name="sweep")
    x, L, wgu, wd = gu.make_layer(wl, T)
    ref, _, _ = gu.run_gpu(x, L, wgu, wd, k, "decode")
    for gw in (1, 2, 4, 16):
        for dw in (1, 3, 16):
            out, _, _ = gu.run_gpu(x, L, wgu, wd, k, "decode", gate_up_warps=gw, down_warps=dw)
            assert torch.equal(out, ref), (gw, dw)


def test_grouped_launch_config_sweep():
    T, H, I, E, k = 200, 512, 256, 12, 4
    wl = gu.custom(T, H, I, E, k, 2.0, name="gsweep")
    x, L, wgu, wd = gu.make_layer(wl, T)
    ref, _, _ = gu.run_gpu(x, L, wgu, wd, k, "grouped")
    for ctas in (1, 7, 64, 300):
        out, _, _ = gu.run_gpu(x, L, wgu, wd, k, "grouped", gemm_ctas=ctas)
        assert torch.equal(out, ref), ctas


def test_auto_path_choice():
    T, H, I, E, k = 80, 256, 128, 8, 2
    wl = gu.custom(T, H, I, E, k, name="auto")
    x, L, wgu, wd = gu.make_layer(wl, T)
    for thr, want in ((0, m.MOE_PATH_GROUPED), (80, m.MOE_PATH_DECODE), (79, m.MOE_PATH_GROUPED)):
        o = m.moe_ffn_opts()
        o.decode_max_tokens = thr
        m.moe_ffn_forward_ex(x, L, wgu, wd, k, opts=o)
        assert o.path_taken == want, (thr, o.path_taken)
        assert o.n_stages == (4 if want == m.MOE_PATH_DECODE else 5)


@pytest.mark.parametrize("T", [1, 6, 200])
def test_plain_forward_and_host_entry_match_ex(T):
    """moe_ffn_forward and moe_ffn_forward_host give moe_ffn_forward_ex's
    bits: host buffers page-locked (small calls read and write them in
    place, large ones copy) and pageable (always copied)."""
    H, I, E, k = 512, 192, 16, 4
    wl = gu.custom(T, H, I, E, k, name="entries")
    x, L, wgu, wd = gu.make_layer(wl, T)
    ref = m.moe_ffn_forward_ex(x, L, wgu, wd, k)
    plain = m.moe_ffn_forward(x, L, wgu, wd, k)
    torch.cuda.synchronize()
    assert torch.equal(plain, ref)
    ws = m.new_workspace(T, H, I, E, k, host=True)
    for pinned in (True, False):
        xh, lh = x.cpu(), L.cpu()
        oh = torch.full((T, H), float("nan"), dtype=torch.float32)
        if pinned:
            xh, lh, oh = xh.pin_memory(), lh.pin_memory(), oh.pin_memory()
        for _ in range(3):
            m.moe_ffn_forward_host(xh, lh, wgu, wd, k, oh, ws)
        torch.cuda.synchronize()
        assert torch.equal(oh, ref.cpu()), pinned


@pytest.mark.parametrize("T,path,stages", [(3, "decode", 1), (8, "decode", 4), (8, "grouped", 5)])
def test_stage_events_time_each_kernel(T, path, stages):
    H, I, E, k = 256, 128, 8, 2
    wl = gu.custom(T, H, I, E, k, name="events")
    x, L, wgu, wd = gu.make_layer(wl, T)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_MAX_STAGES + 1)]
    for e in evs:
        e.record()
    arr = m.stage_event_array(evs)
    o = m.moe_ffn_opts()
    o.path = gu.PATHS[path]
    o.stage_events = m.ctypes.cast(arr, m.ctypes.c_void_p)
    m.moe_ffn_forward_ex(x, L, wgu, wd, k, opts=o)
    torch.cuda.synchronize()
    assert o.n_stages == stages
    for i in range(o.n_stages):
        assert evs[i].elapsed_time(evs[i + 1]) >= 0.0


def test_errors_from_device_pointers():
    """Bad shapes and a short workspace come back as status codes."""
    T, H, I, E, k = 4, 256, 128, 8, 2
    wl = gu.custom(T, H, I, E, k, name="errs")
    x, L, wgu, wd = gu.make_layer(wl, T)
    with pytest.raises(m.MoeFfnError) as ei:
        m.moe_ffn_forward_ex(x, L, wgu, wd, 9)
    assert ei.value.status in (m.MOE_ERR_INVALID_ARG, m.MOE_ERR_UNSUPPORTED_SHAPE)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoeFfnError) as ei:
        m.moe_ffn_forward_ex(x, L, wgu, wd, k, workspace=small)
    assert ei.value.status == m.MOE_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("T,path", [(1, "decode"), (3, "decode"), (8, "decode"), (64, "grouped")])
def test_cuda_graph_replay_matches_eager(T, path):
    """A call captured into a CUDA graph recomputes, on every replay, what an
    eager call gives for the buffers' current contents (the fused decode
    kernel's grid barrier must not reuse a stale epoch on replays)."""
    H, I, E, k = 512, 256, 32, 8
    wl = gu.custom(T, H, I, E, k, 1.0, name="graph")
    inputs = [gu.make_layer(wl, T, call=c)[:2] for c in range(3)]
    _, _, wgu, wd = gu.make_layer(wl, T)
    refs = [gu.run_gpu(x, L, wgu, wd, k, path)[0] for x, L in inputs]
    xb, lb = inputs[0][0].clone(), inputs[0][1].clone()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = m.new_workspace(T, H, I, E, k)
    o = m.moe_ffn_opts()
    o.path = gu.PATHS[path]
    m.moe_ffn_forward_ex(xb, lb, wgu, wd, k, out=out, workspace=ws, opts=o)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_MAX_STAGES + 1)]
    for e in evs:
        e.record()
    arr = m.stage_event_array(evs)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        oc = m.moe_ffn_opts()
        oc.path = gu.PATHS[path]
        oc.stage_events = m.ctypes.cast(arr, m.ctypes.c_void_p)
        m.moe_ffn_forward_ex(xb, lb, wgu, wd, k, out=out, workspace=ws, opts=oc,
                             stream=torch.cuda.current_stream())
    if path == "decode":
        assert oc.path_taken == (m.MOE_PATH_DECODE_FUSED if T <= 4 else m.MOE_PATH_DECODE)
    for r in range(12):
        c = r % 3
        xb.copy_(inputs[c][0])
        lb.copy_(inputs[c][1])
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), refs[c]), (r, c)
    for i in range(oc.n_stages):
        assert evs[i].elapsed_time(evs[i + 1]) >= 0.0


@pytest.mark.parametrize("T,I", [(1, 256), (4, 1024)], ids=["tagged_act", "grid_barrier"])
def test_eager_calls_and_graph_replays_interleaved(T, I):
    """Eager calls and replays of one captured call, interleaved on one
    workspace, each compute their own tokens.  Regression: when a call's
    epoch was a per-launch base plus the device call counter, the replay
    that followed an eager call that followed a replay repeated that eager
    call's epoch, and the fused decode kernel's grid barrier passed on its
    stale arrival words.  T=1 exchanges act through tagged words once the
    workspace is prepared, T=4 with I=1024 (act rows too large to stage)
    always meets at the grid barrier."""
    H, E, k = 512, 32, 8
    wl = gu.custom(T, H, I, E, k, 1.0, name="interleave")
    inputs = [gu.make_layer(wl, T, call=c)[:2] for c in range(6)]
    _, _, wgu, wd = gu.make_layer(wl, T)
    refs = [m.moe_ffn_forward(x, L, wgu, wd, k).cpu() for x, L in inputs]  # keeps no state
    xb, lb = inputs[0][0].clone(), inputs[0][1].clone()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = m.new_workspace(T, H, I, E, k)

    def set_inputs(c):
        xb.copy_(inputs[c][0])
        lb.copy_(inputs[c][1])
        out.fill_(float("nan"))

    set_inputs(0)
    o = m.moe_ffn_opts()
    m.moe_ffn_forward_ex(xb, lb, wgu, wd, k, out=out, workspace=ws, opts=o)
    torch.cuda.synchronize()
    assert o.path_taken == m.MOE_PATH_DECODE_FUSED
    assert torch.equal(out.cpu(), refs[0])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        m.moe_ffn_forward_ex(xb, lb, wgu, wd, k, out=out, workspace=ws, stream=torch.cuda.current_stream())
    steps = ["replay", "eager", "replay", "eager", "eager", "replay", "replay", "eager", "replay"]
    for i, how in enumerate(steps):
        c = (i + 1) % len(inputs)
        set_inputs(c)
        if how == "replay":
            g.replay()
        else:
            m.moe_ffn_forward_ex(xb, lb, wgu, wd, k, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), refs[c]), (i, how)


def test_fused_decode_state_in_a_shared_workspace():
    """One workspace, filled with random bytes first, serves decode calls of
    T = 1..4 (the fused kernel, whose state sits at the same offsets for
    every T) and grouped calls in between.  The first call, and every call
    whose act rows outgrow the prepared tag region, meets at the grid barrier
    and prepares it; the others exchange act through tagged words.  Every
    output matches, bit for bit, a call that keeps no state."""
    H, I, E, k = 512, 256, 32, 8
    seq = [1, 1, 2, 2, 1, 40, 3, 3, 4, 6, 4, 2, 1, 1]
    _, _, wgu, wd = gu.make_layer(gu.custom(1, H, I, E, k, 1.0, name="shared_ws"), 1)
    nbytes = max(m.moe_ffn_workspace_bytes(T, H, I, E, k) for T in seq)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda")
    for step, T in enumerate(seq):
        x, L = synth.make_tokens(gu.custom(T, H, I, E, k, 1.0, name="shared_ws"), T, call=step)
        x, L = x.cuda(), L.cuda()
        ref = m.moe_ffn_forward(x, L, wgu, wd, k).cpu()
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        o = m.moe_ffn_opts()
        m.moe_ffn_forward_ex(x, L, wgu, wd, k, out=out, workspace=ws, opts=o)
        torch.cuda.synchronize()
        assert o.path_taken == (m.MOE_PATH_DECODE_FUSED if T <= 4 else m.MOE_PATH_GROUPED), (T, o.path_taken)
        assert torch.equal(out.cpu(), ref), (step, T)


# Fused decode kernel (T <= 4): tokens that share experts.  Each touched
# expert is streamed once and dotted with every token it serves; the result
# must match the oracle and, bit for bit, the general decode kernels (T > 4
# forced through the decode path uses them) on the same tokens.
@pytest.mark.parametrize("T,share", [(2, "all"), (3, "some"), (4, "all"), (4, "some"), (4, "none")])
def test_fused_decode_shared_experts(T, share):
    H, I, E, k = 512, 256, 32, 8
    wl = gu.custom(T, H, I, E, k, 0.0, name="fused_share")
    x, L, wgu, wd = gu.make_layer(wl, T)
    L = L.clone()
    if share == "all":        # every token picks the same k experts, in the same order
        L[:] = L[0]
    elif share == "some":     # tokens 1.. reuse token 0's two best experts
        L[1:, :] -= 10.0
        top2 = torch.topk(L[0], 2).indices
        L[1:, top2] = L[0, top2] + 20.0
    else:                     # disjoint expert sets
        L[:] = -10.0
        for t in range(T):
            L[t, t * k:(t + 1) * k] = torch.arange(k, 0, -1, dtype=torch.float32, device=L.device)
    out, idx, w = gu.run_gpu(x, L, wgu, wd, k, "decode")
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, L, wgu, wd, k), what=f"T={T} {share}")
    # the same tokens inside a batch of 8 go through the general decode kernels
    x8 = torch.cat([x, x[:1].expand(8 - T, H)]).contiguous()
    L8 = torch.cat([L, L[:1].expand(8 - T, E)]).contiguous()
    out8, idx8, _ = gu.run_gpu(x8, L8, wgu, wd, k, "decode")
    assert torch.equal(idx8[:T], idx)
    assert torch.equal(out8[:T], out)


# Fused decode kernel at the edges of its shape range: H = 64 (most CTAs own
# no output dimension), I = 64, E = 1024 experts, k = 32, and T * k = 64
# assignments (its maximum); and one token on the 2048-hidden geometry (six
# W_down chunks of 21 rows per CTA, experts crossing chunk boundaries),
# I = 1024 and I = 320 (a short last 256-element step).  Compared with the
# oracle and, bit for bit, with the same tokens through the general decode
# kernels.
@pytest.mark.parametrize("T,H,I,E,k", [(1, 64, 64, 1024, 32), (1, 128, 64, 40, 1), (4, 64, 128, 64, 16),
                                       (2, 192, 320, 7, 7), (3, 1024, 64, 256, 8),
                                       (4, 512, 1024, 64, 16),  # act rows too large to stage: read in place
                                       (1, 2048, 768, 32, 8), (1, 512, 1024, 16, 4), (1, 256, 320, 8, 2)])
def test_fused_decode_edges(T, H, I, E, k):
    wl = gu.custom(T, H, I, E, k, 1.0, name="fused_edge")
    x, L, wgu, wd = gu.make_layer(wl, T)
    out, idx, w = gu.run_gpu(x, L, wgu, wd, k, "decode")
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, L, wgu, wd, k), what=str((T, H, I, E, k)))
    x8 = torch.cat([x, x[:1].expand(8 - T, H)]).contiguous()
    L8 = torch.cat([L, L[:1].expand(8 - T, E)]).contiguous()
    out8, idx8, _ = gu.run_gpu(x8, L8, wgu, wd, k, "decode")
    assert torch.equal(idx8[:T], idx)
    assert torch.equal(out8[:T], out)
