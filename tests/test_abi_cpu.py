"""The C-ABI library on the host, without a GPU: it loads, exports every
symbol that include/*.h declares, and rejects bad arguments synchronously
(before any CUDA call), as the header promises."""
import ctypes
import glob
import os
import re

import pytest

from tests.conftest import ROOT

pytestmark = pytest.mark.cpu


@pytest.fixture(scope="module")
def L():
    from mixture_experts_ffn_gate_gb300 import _build, moe_ffn
    _build.build()
    return moe_ffn.lib()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_ffn_forward", "moe_ffn_forward_ex", "moe_ffn_workspace_bytes",
              "moe_ffn_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    from mixture_experts_ffn_gate_gb300 import moe_ffn
    names = declared_functions()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert sorted(moe_ffn.EXPORTED) == names


def test_library_is_in_tree_and_links_no_driver(L):
    from mixture_experts_ffn_gate_gb300 import _build
    assert os.path.realpath(_build.LIB).startswith(os.path.realpath(ROOT))
    # the fixture loaded it although this host may have no GPU driver:
    # libcuda is not a link-time dependency (the TMA encoder is fetched at
    # run time through the CUDA runtime)
    assert L._name == _build.LIB


def test_status_strings(L):
    from mixture_experts_ffn_gate_gb300 import moe_ffn
    for s in range(7):
        assert moe_ffn.moe_ffn_status_string(s) not in ("", "unknown status")
    assert moe_ffn.moe_ffn_status_string(99) == "unknown status"


def test_stage_names(L):
    from mixture_experts_ffn_gate_gb300 import moe_ffn as m
    assert [m.moe_ffn_stage_name(m.MOE_PATH_DECODE, i) for i in range(5)] == \
        ["router", "sort", "decode_gate_up", "decode_down", None]
    assert [m.moe_ffn_stage_name(m.MOE_PATH_DECODE_FUSED, i) for i in range(2)] == ["decode_fused", None]
    assert [m.moe_ffn_stage_name(m.MOE_PATH_GROUPED, i) for i in range(6)] == \
        ["router", "sort", "gemm_gate_up", "gemm_down", "combine", None]
    assert [m.moe_ffn_stage_name(m.MOE_PATH_BACKWARD, i) for i in range(12)] == \
        ["router", "sort", "prep", "gemm_gate_up", "gemm_q", "gemm_dx", "combine", "zero_grads", "wgrad_down",
         "wgrad_gate_up", "dlogits", None]
    assert [m.moe_ffn_stage_name(m.MOE_PATH_TRAIN_FORWARD, i) for i in range(6)] == \
        ["router", "sort", "gemm_gate_up", "gemm_down", "combine", None]
    assert [m.moe_ffn_stage_name(m.MOE_PATH_TRAIN_BACKWARD, i) for i in range(11)] == \
        ["router", "sort", "prep", "gemm_q", "gemm_dx", "combine", "zero_grads", "wgrad_down", "wgrad_gate_up",
         "dlogits", None]
    assert m.moe_ffn_stage_name(m.MOE_PATH_AUTO, 0) is None
    assert m.moe_ffn_stage_name(m.MOE_PATH_DECODE, -1) is None


def test_opts_struct_layout():
    from mixture_experts_ffn_gate_gb300 import moe_ffn as m
    # int32 x 8, two pointers, int32 x 4 (LP64)
    assert ctypes.sizeof(m.moe_ffn_opts) == 64
    assert m.moe_ffn_opts.stage_events.offset == 32
    assert m.moe_ffn_opts.exchange_out.offset == 40
    assert m.moe_ffn_opts.n_stages.offset == 48


def test_workspace_bytes(L):
    ws = L.moe_ffn_workspace_bytes
    assert ws(4, 256, 128, 8, 2) > 0
    assert ws(0, 256, 128, 8, 2) > 0
    assert ws(4, 256, 128, 8, 9) == 0        # k > E
    assert ws(4, 250, 128, 8, 2) == 0        # H % 64
    assert ws(4, 256, 128, 2048, 2) == 0     # E > 1024
    # grows with T
    assert ws(2048, 6144, 2048, 256, 8) > ws(64, 6144, 2048, 256, 8)
    assert L.moe_ffn_host_workspace_bytes(4, 256, 128, 8, 2) > ws(4, 256, 128, 8, 2)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case fails validation first


@pytest.mark.parametrize("case,want", [
    (dict(T=-1), 1), (dict(k=0), 1), (dict(k=9), 1), (dict(E=0), 1),
    (dict(H=200), 2), (dict(I=100), 2), (dict(E=1025, k=2), 2), (dict(k=33, E=64), 2),
    (dict(x=None), 1), (dict(logits=None), 1), (dict(wgu=None), 1), (dict(wd=None), 1),
    (dict(out=None), 1), (dict(x=FAKE + 2), 1), (dict(out=FAKE + 8), 1),
    (dict(workspace=None), 1), (dict(workspace=FAKE + 16), 1),
    (dict(ws_bytes=16), 5), (dict(T=0), 0), (dict(T=0, x=None), 0),
])
def test_argument_checks(L, case, want):
    a = dict(x=FAKE, logits=FAKE, wgu=FAKE, wd=FAKE, T=4, H=256, I=128, E=8, k=2,
             out=FAKE, workspace=FAKE, ws_bytes=1 << 40)
    a.update(case)
    st = L.moe_ffn_forward_ex(a["x"], a["logits"], a["wgu"], a["wd"], a["T"], a["H"], a["I"],
                              a["E"], a["k"], a["out"], a["workspace"], a["ws_bytes"], None,
                              None, None, None)
    assert st == want


def test_bad_opts_rejected(L):
    from mixture_experts_ffn_gate_gb300 import moe_ffn as m
    for field, val in (("path", 3), ("gate_up_warps", 17), ("down_warps", -1), ("gemm_ctas", -2),
                       ("decode_max_tokens", -1), ("test_wait_limit_us", -1),
                       ("test_skip_arrival", -3)):
        o = m.moe_ffn_opts()
        setattr(o, field, val)
        st = L.moe_ffn_forward_ex(FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, FAKE, 1 << 40,
                                  None, None, ctypes.byref(o), None)
        assert st == m.MOE_ERR_INVALID_ARG, field
    o = m.moe_ffn_opts()
    o.reserved_in[0] = 7
    assert L.moe_ffn_forward_ex(FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, FAKE, 1 << 40,
                                None, None, ctypes.byref(o), None) == m.MOE_ERR_INVALID_ARG


def test_plain_forward_checks(L):
    assert L.moe_ffn_forward(None, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, None) == 1
    assert L.moe_ffn_forward(FAKE, FAKE, FAKE, FAKE, 0, 256, 128, 8, 2, FAKE, None) == 0
    assert L.moe_ffn_forward_host(None, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, FAKE, 1 << 40,
                                  None, None) == 1
    assert L.moe_ffn_forward_host(FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, FAKE, 16,
                                  None, None) == 5


def test_product_and_oracle_share_no_code():
    """Neither side imports the other; the CUDA sources include nothing from
    oracle/ and the oracle includes nothing from the package."""
    pkg = os.path.join(ROOT, "mixture_experts_ffn_gate_gb300")
    for f in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if f.endswith((".py", ".cu", ".cuh", ".h")):
            src = open(f).read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
            assert "oracle/" not in src and "moe_oracle" not in src, f
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.*")):
        if f.endswith((".py", ".c", ".h")):
            src = open(f).read()
            assert "mixture_experts_ffn_gate_gb300" not in src and "moe_ffn.h" not in src, f


def test_timeline_build_is_separate_and_exports_its_reader(L):
    """The instrumented build of the fused decode kernel (-DMOE_FUSED_TIMELINE)
    compiles on its own and exports the stamp reader; the product library
    exports no such symbol (its kernels carry no stamps)."""
    from mixture_experts_ffn_gate_gb300 import _build
    path = _build.build_timeline()
    assert os.path.dirname(path) != os.path.dirname(_build.LIB)
    T = ctypes.CDLL(path)
    assert hasattr(T, "moe_ffn_debug_fused_timeline")
    assert not hasattr(L, "moe_ffn_debug_fused_timeline")


@pytest.mark.parametrize("case,want", [
    (dict(x=None), 1), (dict(wr=None), 1), (dict(wgu=None), 1), (dict(out=None), 1),
    (dict(wr=FAKE + 8), 1), (dict(bias=FAKE + 2), 1), (dict(logits=FAKE + 4), 1),
    (dict(workspace=FAKE + 16), 1), (dict(ws_bytes=1024), 5), (dict(k=9), 1), (dict(H=200), 2),
    (dict(T=0), 0), (dict(T=0, x=None), 0), (dict(bias=None), None),
])
def test_router_entry_argument_checks(L, case, want):
    a = dict(x=FAKE, wr=FAKE, bias=FAKE, wgu=FAKE, wd=FAKE, T=4, H=256, I=128, E=8, k=2, out=FAKE,
             workspace=FAKE, ws_bytes=16, logits=None)
    if want is None:   # only checks that a null bias is accepted: stop at the workspace size
        a.update(case)
        want = 5
    else:
        a["ws_bytes"] = 1 << 40 if case.get("ws_bytes") is None else case["ws_bytes"]
        a.update(case)
    st = L.moe_ffn_forward_router(a["x"], a["wr"], a["bias"], a["wgu"], a["wd"], a["T"], a["H"], a["I"],
                                  a["E"], a["k"], a["out"], a["workspace"], a["ws_bytes"], a["logits"],
                                  None, None, None, None)
    assert st == want


def test_router_workspace_bytes(L):
    assert L.moe_ffn_router_workspace_bytes(4, 256, 128, 8, 2) > L.moe_ffn_workspace_bytes(4, 256, 128, 8, 2)
    assert L.moe_ffn_router_workspace_bytes(4, 256, 128, 8, 9) == 0


@pytest.mark.parametrize("case,want", [
    (dict(x=None), 1), (dict(gs=None), 1), (dict(ds=FAKE + 8), 1), (dict(gq=FAKE + 1), 1),
    (dict(logits=None), 1), (dict(workspace=FAKE + 16), 1), (dict(ws_bytes=1024), 5), (dict(k=9), 1),
    (dict(H=200), 2), (dict(T=0), 0), (dict(T=0, x=None), 0),
])
def test_mxfp8_entry_argument_checks(L, case, want):
    a = dict(x=FAKE, logits=FAKE, gq=FAKE, gs=FAKE, dq=FAKE, ds=FAKE, T=4, H=256, I=128, E=8, k=2, out=FAKE,
             workspace=FAKE, ws_bytes=1 << 40)
    a.update(case)
    st = L.moe_ffn_forward_mxfp8(a["x"], a["logits"], a["gq"], a["gs"], a["dq"], a["ds"], a["T"], a["H"], a["I"],
                                 a["E"], a["k"], a["out"], a["workspace"], a["ws_bytes"], None, None, None, None)
    assert st == want


def test_mx_scale_row_bytes_agree():
    from mixture_experts_ffn_gate_gb300 import moe_ffn, synth
    for K in (32, 64, 96, 512, 768, 1536, 2048, 6144, 7168):
        assert moe_ffn.mx_scale_bytes(K) == synth.mx_scale_row_bytes(K) == -(-(K // 32) // 16) * 16


def test_backward_workspace_bytes(L):
    ws = L.moe_ffn_backward_workspace_bytes
    assert ws(4, 256, 128, 8, 2) > 0
    assert ws(4, 256, 128, 8, 9) == 0        # k > E
    assert ws(4, 250, 128, 8, 2) == 0        # H % 64
    assert ws(2048, 6144, 2048, 256, 8) > ws(64, 6144, 2048, 256, 8)
    # the padded rows: T*k assignments plus at most 15 pad rows per touched expert
    n = 2048 * 8
    rows = n + 15 * 256
    assert ws(2048, 6144, 2048, 256, 8) >= rows * (6144 * 2 * 3 + 6144 * 4 + 2048 * 4 * 4)


@pytest.mark.parametrize("case,want", [
    (dict(T=-1), 1), (dict(k=9), 1), (dict(H=200), 2), (dict(E=1025, k=2), 2),
    (dict(x=None), 1), (dict(logits=None), 1), (dict(wgu=None), 1), (dict(wd=None), 1),
    (dict(dout=None), 1), (dict(dx=None), 1), (dict(dlogits=None), 1), (dict(dwgu=None), 1),
    (dict(dwd=None), 1), (dict(dout=FAKE + 4), 1), (dict(dwd=FAKE + 8), 1),
    (dict(workspace=FAKE + 16), 1), (dict(ws_bytes=1024), 5), (dict(T=0, dwgu=None), 1),
])
def test_backward_entry_argument_checks(L, case, want):
    a = dict(x=FAKE, logits=FAKE, wgu=FAKE, wd=FAKE, dout=FAKE, T=4, H=256, I=128, E=8, k=2, dx=FAKE,
             dlogits=FAKE, dwgu=FAKE, dwd=FAKE, workspace=FAKE, ws_bytes=1 << 40)
    a.update(case)
    st = L.moe_ffn_backward(a["x"], a["logits"], a["wgu"], a["wd"], a["dout"], a["T"], a["H"], a["I"], a["E"],
                            a["k"], a["dx"], a["dlogits"], a["dwgu"], a["dwd"], a["workspace"], a["ws_bytes"],
                            None, None)
    assert st == want


def test_backward_rejects_decode_path(L):
    from mixture_experts_ffn_gate_gb300 import moe_ffn as m
    o = m.moe_ffn_opts()
    o.path = m.MOE_PATH_DECODE
    assert L.moe_ffn_backward(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE,
                              1 << 40, ctypes.byref(o), None) == m.MOE_ERR_UNSUPPORTED_SHAPE


def test_train_state_bytes(L):
    for shape in ((4, 256, 128, 8, 2), (2048, 6144, 2048, 256, 8), (4, 250, 128, 8, 2), (4, 256, 128, 8, 9)):
        assert L.moe_ffn_train_state_bytes(*shape) == L.moe_ffn_backward_workspace_bytes(*shape)


@pytest.mark.parametrize("case,want", [
    (dict(T=-1), 1), (dict(k=9), 1), (dict(H=200), 2), (dict(E=1025, k=2), 2),
    (dict(x=None), 1), (dict(logits=None), 1), (dict(wgu=None), 1), (dict(wd=None), 1), (dict(out=None), 1),
    (dict(state=None), 1), (dict(state=FAKE + 16), 1), (dict(state_bytes=1024), 5), (dict(out=FAKE + 4), 1),
    (dict(T=0, wgu=None), 1),
])
def test_forward_train_argument_checks(L, case, want):
    a = dict(x=FAKE, logits=FAKE, wgu=FAKE, wd=FAKE, T=4, H=256, I=128, E=8, k=2, out=FAKE, state=FAKE,
             state_bytes=1 << 40)
    a.update(case)
    st = L.moe_ffn_forward_train(a["x"], a["logits"], a["wgu"], a["wd"], a["T"], a["H"], a["I"], a["E"], a["k"],
                                 a["out"], a["state"], a["state_bytes"], None, None)
    assert st == want


@pytest.mark.parametrize("case,want", [
    (dict(T=-1), 1), (dict(k=9), 1), (dict(H=200), 2), (dict(x=None), 1), (dict(logits=None), 1),
    (dict(wgu=None), 1), (dict(wd=None), 1), (dict(dout=None), 1), (dict(dx=None), 1), (dict(dlogits=None), 1), (dict(dwgu=None), 1),
    (dict(dwd=None), 1), (dict(dwd=FAKE + 8), 1), (dict(state=None), 1), (dict(state=FAKE + 16), 1),
    (dict(state_bytes=1024), 5), (dict(T=0, dwgu=None), 1),
])
def test_backward_train_argument_checks(L, case, want):
    a = dict(x=FAKE, logits=FAKE, wgu=FAKE, wd=FAKE, dout=FAKE, T=4, H=256, I=128, E=8, k=2, dx=FAKE, dlogits=FAKE,
             dwgu=FAKE, dwd=FAKE, state=FAKE, state_bytes=1 << 40)
    a.update(case)
    st = L.moe_ffn_backward_train(a["x"], a["logits"], a["wgu"], a["wd"], a["dout"], a["T"], a["H"], a["I"],
                                  a["E"], a["k"],
                                  a["dx"], a["dlogits"], a["dwgu"], a["dwd"], a["state"], a["state_bytes"], None,
                                  None)
    assert st == want


def test_train_pair_rejects_decode_path(L):
    from mixture_experts_ffn_gate_gb300 import moe_ffn as m
    o = m.moe_ffn_opts()
    o.path = m.MOE_PATH_DECODE
    assert L.moe_ffn_forward_train(FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, FAKE, 1 << 40,
                                   ctypes.byref(o), None) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_ffn_backward_train(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    1 << 40, ctypes.byref(o), None) == m.MOE_ERR_UNSUPPORTED_SHAPE
