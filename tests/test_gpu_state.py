"""The state the fused decode kernel keeps in a workspace between calls, when
calls of different shapes and paths share the workspace, and the give-up
path of its bounded waits.

The fused kernel (T <= 4) exchanges its act rows through epoch-tagged words
in the workspace's tag region without a grid barrier once a barrier call has
cleared that region.  The region's length depends on k and I, and the other
regions of a call follow it, so a call of a smaller k*I writes its routing,
act or staged rows inside a larger shape's region.  Every call therefore
lowers the state's count of prepared words to its own tag capacity.  These
tests check, through ``moe_ffn_opts.exchange_out``, that a fused call after
such a call meets at the barrier again, and that every output equals, bit
for bit, a call that keeps no state (``moe_ffn_forward``).
"""
import pytest
import torch

from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BARRIER, TAGGED = m.EXCHANGE_BARRIER, m.EXCHANGE_TAGGED
FAULT_DECODE_BARRIER = 64 << 8   # fused decode kernel's barrier bit in moe_ffn_device_faults


@pytest.fixture(autouse=True)
def _no_faults_left():
    m.moe_ffn_device_faults(clear=True)
    yield
    assert m.moe_ffn_device_faults(clear=True) == 0, "a kernel's bounded wait gave up"


# Shapes (T, H, I, E, k).  Tag region = min(4k, 64) * I words; a call's
# other regions start at its tag capacity (that rounded up to 32 words).
A = (2, 1024, 512, 32, 4)    # fused, staged act; tag cap 8192, needs 4096
B = (5, 512, 256, 16, 2)     # grouped (AUTO at T=5); tag cap 2048
C = (1, 512, 256, 16, 2)     # fused; tag cap 2048, needs 512
D = (3, 768, 128, 8, 8)      # fused; tag cap 4096, needs 3072
Edec = (6, 1024, 512, 32, 4)  # same k and I as A, general decode kernels
F = (4, 512, 1024, 64, 16)   # fused, act too large to stage: always the barrier
G = (2, 512, 256, 16, 2)     # host entry, pageable buffers (staged in the workspace)

# (shape, path, entry, expected exchange of a fused call or None)
SEQUENCE = [
    (A, "auto", "ex", BARRIER),     # fresh (random) workspace
    (A, "auto", "ex", TAGGED),
    (B, "auto", "ex", None),        # grouped: writes idx, xs, z ... inside A's region
    (A, "auto", "ex", BARRIER),     # so A meets at the barrier again
    (A, "auto", "ex", TAGGED),
    (C, "auto", "ex", TAGGED),      # smaller need, region cleared by A: trusted; lowers it to 2048
    (A, "auto", "ex", BARRIER),
    (D, "auto", "ex", TAGGED),      # 3072 <= 4096 prepared; its cap 4096 keeps them
    (A, "auto", "ex", TAGGED),      # D wrote only tags below 4096
    (Edec, "decode", "ex", None),   # same k, I as A: its regions lie past A's region
    (A, "auto", "ex", TAGGED),
    (F, "auto", "ex", BARRIER),     # reads act in place (past its own cap)
    (A, "auto", "ex", TAGGED),
    (G, "auto", "host", TAGGED),    # staged x / logits / out land inside A's region
    (A, "auto", "ex", BARRIER),
    (A, "auto", "ex", TAGGED),
]


def _layer(shape, call):
    T, H, I, E, k = shape
    wl = gu.custom(T, H, I, E, k, 0.5, name="state_%d_%d_%d_%d" % (H, I, E, k))
    wgu, wd = synth.make_weights(wl)
    x, L = synth.make_tokens(wl, T, call=call)
    return x.cuda(), L.cuda(), wgu.cuda(), wd.cuda()


def _ws_bytes(shapes):
    return max(max(m.moe_ffn_workspace_bytes(*s), m.moe_ffn_host_workspace_bytes(*s)) for s in shapes)


def test_exchange_mode_and_bits_across_shapes_on_one_workspace():
    """Calls of five shapes (fused decode with staged and in-place act,
    general decode, grouped, host entry) share one workspace that starts as
    random bytes.  Every output equals a stateless call's bit for bit, and
    every fused call whose scratch another call has overwritten meets at the
    grid barrier (exchange_out == 1) before it trusts the tags again."""
    shapes = sorted({s for s, *_ in SEQUENCE})
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    ws = torch.randint(0, 256, (_ws_bytes(shapes),), dtype=torch.uint8, device="cuda", generator=g)
    mode = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step, (shape, path, entry, want) in enumerate(SEQUENCE):
        T, H, I, E, k = shape
        x, L, wgu, wd = _layer(shape, call=step)
        o = m.moe_ffn_opts()
        o.path = {"auto": m.MOE_PATH_AUTO, "decode": m.MOE_PATH_DECODE}[path]
        # a call that keeps no state, on the same path (the two paths are
        # each deterministic but not bitwise equal to each other)
        if path == "auto":
            ref = m.moe_ffn_forward(x, L, wgu, wd, k).cpu()
        else:
            ro = m.moe_ffn_opts()
            ro.path = o.path
            ref = m.moe_ffn_forward_ex(x, L, wgu, wd, k, opts=ro).cpu()   # a fresh workspace
        o.exchange_out = mode.data_ptr()
        mode.fill_(0)
        if entry == "ex":
            out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
            m.moe_ffn_forward_ex(x, L, wgu, wd, k, out=out, workspace=ws, opts=o)
            torch.cuda.synchronize()
            got = out.cpu()
        else:
            oh = torch.full((T, H), float("nan"), dtype=torch.float32)
            m.moe_ffn_forward_host(x.cpu(), L.cpu(), wgu, wd, k, oh, ws, opts=o)
            torch.cuda.synchronize()
            got = oh
        assert torch.equal(got, ref), (step, shape)
        fused = o.path_taken == m.MOE_PATH_DECODE_FUSED
        assert fused == (want is not None), (step, shape, o.path_taken)
        assert int(mode.item()) == (want if fused else 0), (step, shape, int(mode.item()))


def test_noalloc_array_across_shapes_matches_stateless_calls():
    """The same sequence (all but the host entry) through
    moe_ffn_forward_noalloc, whose fixed array keeps the state of every
    shape: bit-identical to stateless calls."""
    for step, (shape, path, entry, _) in enumerate(SEQUENCE):
        if entry != "ex" or path != "auto":
            continue
        T, H, I, E, k = shape
        x, L, wgu, wd = _layer(shape, call=100 + step)
        ref = m.moe_ffn_forward(x, L, wgu, wd, k)
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        m.moe_ffn_forward_noalloc(x, L, wgu, wd, k, out=out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), (step, shape)


def test_cleared_state_bytes_discard_the_state():
    """Zeroing a workspace's first MOE_FFN_WORKSPACE_STATE_BYTES bytes (the
    rule for memory that held other data in between) sends the next fused
    call through the barrier, with the same bits."""
    T, H, I, E, k = A
    x, L, wgu, wd = _layer(A, call=0)
    ws = m.new_workspace(T, H, I, E, k)
    mode = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = m.moe_ffn_opts()
    o.exchange_out = mode.data_ptr()
    seen = []
    outs = []
    for i in range(4):
        if i == 2:
            ws[:m.MOE_FFN_WORKSPACE_STATE_BYTES].zero_()
        outs.append(m.moe_ffn_forward_ex(x, L, wgu, wd, k, workspace=ws, opts=o).clone())
        torch.cuda.synchronize()
        seen.append(int(mode.item()))
    assert seen == [BARRIER, TAGGED, BARRIER, TAGGED]
    for r in outs[1:]:
        assert torch.equal(r, outs[0])


@pytest.mark.parametrize("shape", [(1, 512, 256, 32, 8), (3, 1024, 512, 32, 4)], ids=["T1", "T3"])
def test_bounded_wait_gives_up_and_the_next_call_is_correct(shape):
    """A fused call whose last CTA skips its arrival at the grid barrier (a
    test hook; nothing faults) waits out its bounded waits (20 ms here),
    sets the fused decode barrier bit in the device fault word and writes no
    output.  The next call on the same workspace is bit-correct, and the one
    after it exchanges through tags again."""
    T, H, I, E, k = shape
    x, L, wgu, wd = _layer(shape, call=3)
    ref = m.moe_ffn_forward(x, L, wgu, wd, k).cpu()
    ws = m.new_workspace(T, H, I, E, k)
    mode = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.moe_ffn_forward_ex(x, L, wgu, wd, k, workspace=ws)           # prepares the tag region
    torch.cuda.synchronize()
    assert m.moe_ffn_device_faults(clear=True) == 0

    o = m.moe_ffn_opts()
    o.test_skip_arrival = 1
    o.test_wait_limit_us = 20000
    o.exchange_out = mode.data_ptr()
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    m.moe_ffn_forward_ex(x, L, wgu, wd, k, out=out, workspace=ws, opts=o)
    torch.cuda.synchronize()
    assert o.path_taken == m.MOE_PATH_DECODE_FUSED
    assert int(mode.item()) == BARRIER            # the hook forces the barrier
    faults = m.moe_ffn_device_faults(clear=True)
    assert faults & FAULT_DECODE_BARRIER, hex(faults)
    assert faults & 0xff == 0, hex(faults)        # no grouped-GEMM bit
    assert torch.isnan(out).all()                 # the call gave up before writing

    for want in (None, TAGGED):
        o = m.moe_ffn_opts()
        o.exchange_out = mode.data_ptr()
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        m.moe_ffn_forward_ex(x, L, wgu, wd, k, out=out, workspace=ws, opts=o)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), ref)
        if want is not None:
            assert int(mode.item()) == want
    assert m.moe_ffn_device_faults(clear=True) == 0
