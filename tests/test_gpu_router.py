"""The layer with its router projection inside the call
(moe_ffn_forward_router): logits bit-exact against the oracle's exactly
rounded projection, routing indices bit-exact, outputs within the parity
tolerance, and outputs bit-identical to the logits entry point given the
same logits -- on the fused decode kernel (T <= 4), on the general decode
kernels and on the grouped path."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_faults():
    m.moe_ffn_device_faults(clear=True)
    yield
    assert m.moe_ffn_device_faults(clear=True) == 0, "a kernel's bounded wait gave up"


def _layer(T, H, I, E, k, bias_var, call=0, name="router_layer"):
    wl = gu.custom(T, H, I, E, k, bias_var, name=name)
    wgu, wd = synth.make_weights(wl)
    wr = synth.make_router(wl)
    x, _ = synth.make_tokens(wl, T, call=call)
    b = synth.make_bias(wl) if bias_var else None
    return x.cuda(), wr.cuda(), (None if b is None else b.cuda()), wgu.cuda(), wd.cuda()


def _run(x, wr, b, wgu, wd, k, path=m.MOE_PATH_AUTO, workspace=None):
    T, E = x.shape[0], wr.shape[0]
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    o = m.moe_ffn_opts()
    o.path = path
    out = m.moe_ffn_forward_router(x, wr, b, wgu, wd, k, logits=logits, topk_idx=idx, topk_w=w, opts=o,
                                   workspace=workspace)
    torch.cuda.synchronize()
    return out.cpu(), logits.cpu(), idx.cpu(), w.cpu(), o.path_taken


def _oracle_logits(x, wr, b):
    return oracle.router_logits(synth.bf16_bits(x), synth.bf16_bits(wr),
                                None if b is None else b.cpu().numpy())


# (T, H, I, E, k, bias variance, path): the fused decode kernel for T <= 4,
# the general decode kernels (T = 5 forced) and the grouped path.
CASES = [
    (1, 256, 128, 8, 2, 0.0, "auto"), (2, 512, 256, 32, 4, 0.5, "auto"), (3, 320, 192, 5, 3, 1.0, "auto"),
    (4, 1024, 256, 64, 8, 0.5, "auto"), (1, 64, 64, 1024, 32, 1.0, "auto"),
    (5, 512, 256, 16, 4, 0.5, "decode"), (40, 384, 192, 12, 3, 0.5, "grouped"), (40, 384, 192, 12, 3, 0.0, "auto"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_H%d_I%d_E%d_k%d_%s" % (c[:5] + (c[6],)))
def test_router_entry_against_oracle(case):
    T, H, I, E, k, bv, path = case
    x, wr, b, wgu, wd = _layer(T, H, I, E, k, bv)
    out, logits, idx, w, taken = _run(x, wr, b, wgu, wd, k, gu.PATHS.get(path, m.MOE_PATH_AUTO))
    if T <= 4 and path == "auto":
        assert taken == m.MOE_PATH_DECODE_FUSED
    want_logits = _oracle_logits(x, wr, b)
    assert np.array_equal(logits.numpy(), want_logits), "logits differ from the exactly rounded projection"
    ref = gu.oracle_ref(x, torch.as_tensor(want_logits).cuda(), wgu, wd, k)
    gu.assert_accepted(out, idx, w, *ref, what=str(case))
    # the logits entry point on the same logits and path gives the same bits
    o = m.moe_ffn_opts()
    o.path = gu.PATHS.get(path, m.MOE_PATH_AUTO)
    same = m.moe_ffn_forward_ex(x, torch.as_tensor(want_logits).cuda(), wgu, wd, k, opts=o)
    torch.cuda.synchronize()
    assert torch.equal(same.cpu(), out)


@pytest.mark.parametrize("name,T", [("decode_h2048_i768_e128_k8", 1), ("decode_h2048_i768_e128_k8", 2),
                                    ("decode_h4096_i1536_e128_k8_bias", 4)], ids=lambda v: str(v))
def test_router_entry_full_size(name, T):
    wl = synth.WORKLOADS[name]
    wgu, wd = synth.make_weights(wl, device="cuda")
    wr = synth.make_router(wl, device="cuda")
    b = synth.make_bias(wl).cuda()
    x, _ = synth.make_tokens(wl, T, call=5, device="cuda")
    out, logits, idx, w, taken = _run(x, wr, b, wgu, wd, wl.k)
    assert taken == m.MOE_PATH_DECODE_FUSED
    want_logits = _oracle_logits(x, wr, b)
    assert np.array_equal(logits.numpy(), want_logits)
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, torch.as_tensor(want_logits).cuda(), wgu, wd, wl.k),
                       what=f"{name} T={T}")


def test_router_entry_ties_from_duplicated_rows():
    """Duplicated router rows give exactly equal logits; the lower expert
    index wins, on the fused kernel and on the general path alike."""
    T, H, I, E, k = 3, 256, 128, 16, 5
    x, wr, _, wgu, wd = _layer(T, H, I, E, k, 0.0, name="router_ties")
    wr = wr.clone()
    wr[9] = wr[2]
    wr[14] = wr[2]
    wr[5] = wr[11]
    b = torch.zeros(E, dtype=torch.float32, device="cuda")
    b[[2, 9, 14]] = 3.0      # push the duplicated experts into every token's top k
    out, logits, idx, w, taken = _run(x, wr, b, wgu, wd, k)
    assert taken == m.MOE_PATH_DECODE_FUSED
    assert torch.equal(logits[:, 2], logits[:, 9]) and torch.equal(logits[:, 2], logits[:, 14])
    want_logits = _oracle_logits(x, wr, b)
    assert np.array_equal(logits.numpy(), want_logits)
    gu.assert_accepted(out, idx, w, *gu.oracle_ref(x, torch.as_tensor(want_logits).cuda(), wgu, wd, k),
                       what="ties")
    for t in range(T):
        sel = idx[t].tolist()
        assert sel.index(2) < sel.index(9) < sel.index(14)
    x8 = torch.cat([x, x[:1].expand(8 - T, H)]).contiguous()
    out8, logits8, idx8, _, taken8 = _run(x8, wr, b, wgu, wd, k, m.MOE_PATH_DECODE)
    assert taken8 == m.MOE_PATH_DECODE
    assert torch.equal(logits8[:T], logits) and torch.equal(idx8[:T], idx) and torch.equal(out8[:T], out)


def test_router_entry_reused_workspace_and_graph_replay():
    """One workspace, eager calls and replays of a captured call over
    changing tokens: every output equals a call on a fresh workspace (the
    tagged logit words of earlier calls never pass for this call's)."""
    T, H, I, E, k = 1, 512, 256, 32, 8
    x0, wr, b, wgu, wd = _layer(T, H, I, E, k, 0.5, name="router_reuse")
    xs = [_layer(T, H, I, E, k, 0.5, call=c, name="router_reuse")[0] for c in range(6)]
    refs = [m.moe_ffn_forward_router(xc, wr, b, wgu, wd, k).cpu() for xc in xs]   # fresh workspaces
    torch.cuda.synchronize()
    ws = m.new_router_workspace(T, H, I, E, k)
    xb = xs[0].clone()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    m.moe_ffn_forward_router(xb, wr, b, wgu, wd, k, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), refs[0])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        m.moe_ffn_forward_router(xb, wr, b, wgu, wd, k, out=out, workspace=ws,
                                 stream=torch.cuda.current_stream())
    for i, how in enumerate(["replay", "eager", "replay", "replay", "eager", "eager", "replay"]):
        c = (i + 1) % len(xs)
        xb.copy_(xs[c])
        out.fill_(float("nan"))
        if how == "replay":
            g.replay()
        else:
            m.moe_ffn_forward_router(xb, wr, b, wgu, wd, k, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), refs[c]), (i, how)


def test_router_entry_errors():
    T, H, I, E, k = 2, 256, 128, 8, 2
    x, wr, b, wgu, wd = _layer(T, H, I, E, k, 0.5)
    small = torch.empty(m.moe_ffn_workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoeFfnError) as ei:   # the logits entry's size is not enough
        m.moe_ffn_forward_router(x, wr, b, wgu, wd, k, workspace=small)
    assert ei.value.status == m.MOE_ERR_WORKSPACE_TOO_SMALL


def test_router_entry_fresh_workspaces_at_reused_addresses():
    """Calls that each get a fresh workspace from torch's caching allocator
    (the same addresses again and again, state bytes zeroed, so every call
    counter starts at zero): no call may take the tagged logit words an
    earlier call left at that address for its own.  Regression: with the
    epoch alone tagging those words, three of six such calls routed on the
    previous call's logits."""
    T, H, I, E, k = 1, 512, 256, 32, 8
    _, wr, b, wgu, wd = _layer(T, H, I, E, k, 0.5, name="router_fresh")
    for c in range(8):
        x = _layer(T, H, I, E, k, 0.5, call=c, name="router_fresh")[0]
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        out = m.moe_ffn_forward_router(x, wr, b, wgu, wd, k, logits=logits)   # a fresh workspace
        same = m.moe_ffn_forward_ex(x, logits, wgu, wd, k)
        torch.cuda.synchronize()
        assert np.array_equal(logits.cpu().numpy(), _oracle_logits(x, wr, b)), c
        assert torch.equal(out, same), c
