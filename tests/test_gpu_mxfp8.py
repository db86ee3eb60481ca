"""The layer with MXFP8 expert weights (moe_ffn_forward_mxfp8: the fused
decode kernel's MX instantiation for T <= 4, the general decode kernels' MX
instantiations up to 8 tokens (and up to 64 when MOE_PATH_DECODE is
forced), the tensor-core grouped GEMMs' MX kinds beyond) against the oracle on the exactly dequantised
weights: routing indices bit-exact, routing weights and outputs within the
parity tolerance (tests/gpu_util.py), at small ragged shapes, at the decode
workloads' full sizes, with signed zeros, subnormal codes and spread scales,
across calls on one workspace (both act exchanges) and in CUDA-graph replays,
bit-identical across runs and grid widths on the grouped path; plus the
argument checks."""
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


def _layer(wl, T, call=0):
    gq, gs, dq, ds = synth.make_weights_mxfp8(wl, device="cuda")
    bias = synth.make_bias(wl)
    x, L = synth.make_tokens(wl, T, call=call, bias=bias)
    return x.cuda(), L.cuda(), gq, gs, dq, ds


def _run(x, L, gq, gs, dq, ds, k, workspace=None, opts=None, path=None):
    T = x.shape[0]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    o = opts or m.moe_ffn_opts()
    if path is not None:
        o.path = path
    out = m.moe_ffn_forward_mxfp8(x, L, gq, gs, dq, ds, k, topk_idx=idx, topk_w=w, opts=o, workspace=workspace)
    torch.cuda.synchronize()
    if path == m.MOE_PATH_DECODE:
        assert o.path_taken in (m.MOE_PATH_DECODE_FUSED, m.MOE_PATH_DECODE)
    else:
        want = m.MOE_PATH_DECODE_FUSED if T <= 4 else m.MOE_PATH_DECODE if T <= 8 else m.MOE_PATH_GROUPED
        assert o.path_taken == (m.MOE_PATH_GROUPED if path == m.MOE_PATH_GROUPED else want)
    return out.cpu(), idx.cpu(), w.cpu()


def _oracle(x, L, gq, gs, dq, ds, k):
    """The oracle on the selected experts' codes and scales only."""
    Ln = L.cpu().numpy()
    idx, _ = oracle.route(Ln, k)
    used = np.unique(idx)
    emap = -np.ones(Ln.shape[1], np.int32)
    emap[used] = np.arange(len(used), dtype=np.int32)
    sel = torch.as_tensor(used, dtype=torch.long, device=gq.device)
    pick = lambda t: t.index_select(0, sel).cpu().numpy()
    return oracle.forward_mxfp8(synth.bf16_bits(x), Ln, pick(gq), pick(gs), pick(dq), pick(ds), k, expert_map=emap)


# (T, H, I, E, k, bias variance): ragged lane coverage (H or I not a
# multiple of 512), scale rows with padding (I = 192: 6 scales in 16 bytes),
# many experts with k = 32, one to four tokens (fused kernel) and more
# (grouped path: ragged 128-row tiles with H = 576 or I = 192 / 320, experts
# with several 64-row chunks, a skewed load, one expert)
SMALL = [(1, 256, 128, 8, 2, 0.0), (2, 576, 192, 16, 4, 0.5), (3, 1024, 320, 32, 8, 1.0),
         (4, 512, 192, 12, 3, 0.5), (1, 64, 64, 1024, 32, 1.0), (4, 2048, 768, 128, 8, 0.0),
         (5, 576, 192, 16, 4, 0.5), (13, 1024, 320, 8, 3, 1.0), (64, 512, 256, 12, 2, 4.0),
         (300, 256, 128, 4, 2, 0.0), (97, 640, 320, 24, 5, 2.0), (40, 128, 64, 1, 1, 0.0)]


@pytest.mark.parametrize("T,H,I,E,k,bv", SMALL)
def test_mxfp8_parity_small(T, H, I, E, k, bv):
    wl = gu.custom(T, H, I, E, k, bv, name="mx_small")
    x, L, gq, gs, dq, ds = _layer(wl, T)
    out, idx, w = _run(x, L, gq, gs, dq, ds, k)
    gu.assert_accepted(out, idx, w, *_oracle(x, L, gq, gs, dq, ds, k), what=f"mxfp8 {T, H, I, E, k}")


@pytest.mark.parametrize("T,H,I,E,k,bv", [(5, 576, 192, 16, 4, 0.5), (13, 1024, 320, 8, 3, 1.0),
                                          (64, 512, 256, 12, 2, 4.0)])
def test_mxfp8_parity_general_decode(T, H, I, E, k, bv):
    """The general decode kernels' MX instantiations (MOE_PATH_DECODE)."""
    wl = gu.custom(T, H, I, E, k, bv, name="mx_small")
    x, L, gq, gs, dq, ds = _layer(wl, T)
    out, idx, w = _run(x, L, gq, gs, dq, ds, k, path=m.MOE_PATH_DECODE)
    gu.assert_accepted(out, idx, w, *_oracle(x, L, gq, gs, dq, ds, k), what=f"mxfp8 decode {T, H, I, E, k}")


def test_mxfp8_grouped_bit_identical_across_runs_and_widths():
    wl = gu.custom(200, 512, 256, 16, 4, 1.0, name="mx_det")
    x, L, gq, gs, dq, ds = _layer(wl, 200)
    ref = _run(x, L, gq, gs, dq, ds, 4)[0]
    for ctas in (0, 37, 1):
        o = m.moe_ffn_opts()
        o.gemm_ctas = ctas
        assert torch.equal(_run(x, L, gq, gs, dq, ds, 4, opts=o)[0], ref), ctas


@pytest.mark.parametrize("name,T", [("decode_h2048_i768_e128_k8", 1), ("decode_h2048_i768_e128_k8", 2),
                                    ("decode_h4096_i1536_e128_k8_bias", 4), ("decode_h7168_i2048_e384_k8_bias", 1),
                                    ("decode_h4096_i1536_e128_k8_bias", 16), ("decode_h7168_i2048_e384_k8_bias", 8),
                                    ("decode_h4096_i1536_e128_k8_bias", 64), ("decode_h7168_i2048_e384_k8_bias", 32)])
def test_mxfp8_parity_full_size(name, T):
    wl = synth.WORKLOADS[name]
    x, L, gq, gs, dq, ds = _layer(wl, T, call=7)
    out, idx, w = _run(x, L, gq, gs, dq, ds, wl.k)
    gu.assert_accepted(out, idx, w, *_oracle(x, L, gq, gs, dq, ds, wl.k), what=f"mxfp8 {name} T={T}")


@pytest.mark.parametrize("T,spread", [(3, 12), (40, 12), (40, 40)])
def test_mxfp8_signed_zeros_subnormal_codes_and_spread_scales(T, spread):
    """+-0 and subnormal codes, scales moved by up to +-spread: T = 3 takes
    the fused kernel, T = 40 the grouped path, whose conversion multiplies by
    2^(min(s, 127) - 15) and 2^(max(s, 127) - 127) (the spread of 40 takes
    scales past 142, where 2^(s - 15) itself is no BF16 number)."""
    H, I, E, k = 512, 256, 16, 4
    wl = gu.custom(T, H, I, E, k, 0.5, name="mx_edges")
    x, L, gq, gs, dq, ds = _layer(wl, T)
    g = torch.Generator(device="cpu").manual_seed(11)
    for q in (gq, dq):
        r = torch.randint(0, 256, q.shape, generator=g, dtype=torch.int32)
        codes = q.cpu().to(torch.int32)
        # a quarter of the codes replaced by +-0 and subnormals (exponent field 0)
        sub = torch.where(r % 2 == 0, r % 8, 0x80 | (r % 8))
        codes = torch.where(r % 4 == 0, sub, codes)
        q.copy_(codes.to(torch.uint8).cuda())
    for s in (gs, ds):
        r = torch.randint(-spread, spread + 1, s.shape, generator=g, dtype=torch.int32)
        s.copy_((s.cpu().to(torch.int32) + r).clamp(1, 254).to(torch.uint8).cuda())
    if spread > 30:
        assert int(gs.max()) > 142 or int(ds.max()) > 142
    out, idx, w = _run(x, L, gq, gs, dq, ds, k)
    gu.assert_accepted(out, idx, w, *_oracle(x, L, gq, gs, dq, ds, k), what=f"mxfp8 edge codes T={T} spread={spread}")


def test_mxfp8_workspace_reuse_exchanges_and_graph_replay():
    """One workspace across token counts: the first fused call meets at the
    grid barrier, later ones exchange tagged words; eager calls and a CUDA
    graph of the same calls give the fresh-workspace bits."""
    wl = synth.WORKLOADS["decode_h2048_i768_e128_k8"]
    gq, gs, dq, ds = synth.make_weights_mxfp8(wl, device="cuda")
    batches = [synth.make_tokens(wl, T, call=c) for c, T in enumerate([1, 2, 4, 1, 3, 2])]
    batches = [(x.cuda(), L.cuda()) for x, L in batches]
    refs = [m.moe_ffn_forward_mxfp8(x, L, gq, gs, dq, ds, wl.k).cpu() for x, L in batches]
    ws = m.new_workspace(4, wl.H, wl.I, wl.E, wl.k)
    mode = torch.zeros(1, dtype=torch.int32, device="cuda")
    seen = []
    for (x, L), ref in zip(batches, refs):
        o = m.moe_ffn_opts()
        o.exchange_out = mode.data_ptr()
        out = m.moe_ffn_forward_mxfp8(x, L, gq, gs, dq, ds, wl.k, workspace=ws, opts=o)
        torch.cuda.synchronize()
        seen.append(int(mode.item()))
        assert torch.equal(out.cpu(), ref)
    assert seen[0] == m.EXCHANGE_BARRIER and m.EXCHANGE_TAGGED in seen[1:]
    outs = [torch.empty((x.shape[0], wl.H), dtype=torch.float32, device="cuda") for x, _ in batches]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        for (x, L), o in zip(batches, outs):
            m.moe_ffn_forward_mxfp8(x, L, gq, gs, dq, ds, wl.k, out=o, workspace=ws, stream=s)
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for o, ref in zip(outs, refs):
            assert torch.equal(o.cpu(), ref)


def test_mxfp8_argument_checks():
    T, H, I, E, k = 2, 256, 128, 8, 2
    wl = gu.custom(T, H, I, E, k, name="mx_args")
    x, L, gq, gs, dq, ds = _layer(wl, T)
    lib = m.lib()
    ws = m.new_workspace(8, H, I, E, k)
    out = torch.empty((8, H), dtype=torch.float32, device="cuda")
    p = lambda t: t.data_ptr()
    nbytes = ws.numel()

    def call(x_=x, gs_=p(gs), T_=T, ws_=p(ws), n_=nbytes, o=None):
        return lib.moe_ffn_forward_mxfp8(p(x_), p(L), p(gq), gs_, p(dq), p(ds), T_, H, I, E, k, p(out), ws_, n_,
                                         None, None, o, None)

    assert call() == m.MOE_OK
    torch.cuda.synchronize()
    assert call(gs_=p(gs) + 1) == m.MOE_ERR_INVALID_ARG           # misaligned scales
    assert call(gs_=None) == m.MOE_ERR_INVALID_ARG
    assert call(n_=1024) == m.MOE_ERR_WORKSPACE_TOO_SMALL
    xb = torch.cat([x] * 33)
    Lb = torch.cat([L] * 33)
    wsb = m.new_workspace(65, H, I, E, k)
    outb = torch.empty((66, H), dtype=torch.float32, device="cuda")
    o = m.moe_ffn_opts()
    o.path = m.MOE_PATH_DECODE   # the general decode kernels take at most 64 tokens
    assert lib.moe_ffn_forward_mxfp8(p(xb), p(Lb), p(gq), p(gs), p(dq), p(ds), 65, H, I, E, k, p(outb), p(wsb),
                                     wsb.numel(), None, None, m.ctypes.byref(o), None) == m.MOE_ERR_UNSUPPORTED_SHAPE
    o = m.moe_ffn_opts()         # the grouped path takes them
    assert lib.moe_ffn_forward_mxfp8(p(xb), p(Lb), p(gq), p(gs), p(dq), p(ds), 65, H, I, E, k, p(outb), p(wsb),
                                     wsb.numel(), None, None, m.ctypes.byref(o), None) == m.MOE_OK
    torch.cuda.synchronize()
    assert o.path_taken == m.MOE_PATH_GROUPED
    o = m.moe_ffn_opts()
    o.path = m.MOE_PATH_GROUPED
    assert call(o=m.ctypes.byref(o)) == m.MOE_OK
    torch.cuda.synchronize()
    assert o.path_taken == m.MOE_PATH_GROUPED
    assert lib.moe_ffn_forward_mxfp8(p(x), p(L), p(gq), p(gs), p(dq), p(ds), 0, H, I, E, k, p(out), p(ws), nbytes,
                                     None, None, None, None) == m.MOE_OK                        # T = 0
