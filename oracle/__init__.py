"""FP64 CPU oracle for the routed MoE SwiGLU FFN forward pass.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product (the CUDA
library and its Python binding) never imports this package, and this package
never imports the product: the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, IEEE double, no
``-ffast-math``).  This module only compiles it with gcc and marshals numpy
arrays to it.  MXFP8 expert weights (``mxfp8.py``) are decoded and
dequantised exactly into BF16 numbers before they reach it.  BF16 tensors travel as their raw 16-bit patterns (numpy
``uint16``), so the oracle reads exactly the bits the GPU reads.

What each step computes, and the passage it follows, is written at the top of
``moe_oracle.c``.  The router projection that produces the logits from the
token activations (``router.py``, plain numpy and ``math.fsum``) is the one
step written in Python: its definition is an exactly rounded sum.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")

STATUS = {0: "ok", 1: "invalid argument", 2: "out of memory",
          3: "a selected expert has no weights in the expert map"}

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
             "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra"]


def compile_source(src: str, out: str) -> str:
    """gcc one oracle C source into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/libmoe_oracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a, name):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name} must hold raw bf16 bits as uint16, got {a.dtype}")
    return a


class Oracle:
    """The oracle library at ``lib_path`` (default: the committed source)."""

    def __init__(self, lib_path: str | None = None):
        lib = ctypes.CDLL(lib_path or build())
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_route.argtypes = [vp, i64, i64, i64, vp, vp]
        lib.oracle_forward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64,
                                       i64, i64, vp, vp, vp, ctypes.c_int]
        lib.oracle_expert_ffn.argtypes = [vp, vp, vp, i64, i64, vp]
        for f in (lib.oracle_route, lib.oracle_forward, lib.oracle_expert_ffn):
            f.restype = ctypes.c_int
        self._lib = lib

    @staticmethod
    def _check(status, what):
        if status != 0:
            raise RuntimeError(f"oracle {what} failed: {STATUS.get(status, status)}")

    def route(self, logits: np.ndarray, k: int):
        """Top-k selection and renormalised softmax weights for every token.

        logits: float32 [T, E].  Returns (idx int32 [T, k], w float64 [T, k]).
        """
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float64)
        self._check(self._lib.oracle_route(_ptr(logits), T, E, k, _ptr(idx),
                                           _ptr(w)), "route")
        return idx, w

    def expert_ffn(self, x_row, wgu_e, wd_e):
        """One expert on one token: W_down_e . (silu(W_gate_e x) * (W_up_e x)).

        x_row uint16 [H]; wgu_e uint16 [2I, H]; wd_e uint16 [H, I] (bf16
        bits).  Returns float64 [H].
        """
        x_row, wgu_e, wd_e = _u16(x_row, "x"), _u16(wgu_e, "wgu"), _u16(wd_e, "wd")
        H = x_row.shape[0]
        I = wgu_e.shape[0] // 2
        assert wgu_e.shape == (2 * I, H) and wd_e.shape == (H, I)
        y = np.empty(H, np.float64)
        self._check(self._lib.oracle_expert_ffn(_ptr(x_row), _ptr(wgu_e),
                                                _ptr(wd_e), H, I, _ptr(y)),
                    "expert_ffn")
        return y

    def forward(self, x, logits, wgu, wd, k: int, *, expert_map=None,
                nthreads: int | None = None):
        """The whole layer in FP64.

        x uint16 [T, H]; logits float32 [T, E]; wgu uint16 [Eb, 2I, H];
        wd uint16 [Eb, H, I].  With ``expert_map`` (int32 [E], -1 = absent)
        the weight arrays hold only the blocks that the map names, so a caller
        can pass just the experts its tokens select.  Returns
        (out float64 [T, H], idx int32 [T, k], w float64 [T, k]).
        """
        x, wgu, wd = _u16(x, "x"), _u16(wgu, "wgu"), _u16(wd, "wd")
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, H = x.shape
        E = logits.shape[1]
        I = wgu.shape[1] // 2
        assert logits.shape[0] == T and wgu.shape[1:] == (2 * I, H)
        assert wd.shape[1:] == (H, I) and wd.shape[0] == wgu.shape[0]
        if expert_map is None:
            assert wgu.shape[0] == E
        else:
            expert_map = np.ascontiguousarray(expert_map, dtype=np.int32)
            assert expert_map.shape == (E,)
        if nthreads is None:
            nthreads = len(os.sched_getaffinity(0))
        out = np.empty((T, H), np.float64)
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float64)
        self._check(self._lib.oracle_forward(
            _ptr(x), _ptr(logits), _ptr(wgu), _ptr(wd), _ptr(expert_map), T, H,
            I, E, k, _ptr(out), _ptr(idx), _ptr(w), int(nthreads)), "forward")
        return out, idx, w


_default = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
    return _default


def route(logits, k):
    return default().route(logits, k)


def expert_ffn(x_row, wgu_e, wd_e):
    return default().expert_ffn(x_row, wgu_e, wd_e)


def forward(x, logits, wgu, wd, k, **kw):
    return default().forward(x, logits, wgu, wd, k, **kw)


def router_logits(x, w_router, bias=None):
    """logits float32 [T, E] = round_f32(exact x . W_r^T + b); see router.py."""
    from .router import router_logits as f
    return f(x, w_router, bias)


def forward_router(x, w_router, bias, wgu, wd, k, **kw):
    """The layer from the token activations and the router weights: the
    router projection, then the layer on its logits.  Returns (out, idx, w,
    logits)."""
    logits = router_logits(x, w_router, bias)
    out, idx, w = forward(x, logits, wgu, wd, k, **kw)
    return out, idx, w, logits


def forward_mxfp8(x, logits, wgu_q, wgu_s, wd_q, wd_s, k, **kw):
    """The layer with MXFP8 expert weights (codes uint8 [Eb, 2I, H] and
    [Eb, H, I], scales uint8 [Eb, 2I, Hs] and [Eb, H, Is]; see mxfp8.py):
    the weights dequantised exactly, then the BF16 layer's definition.
    Returns (out, idx, w)."""
    from .mxfp8 import dequantize_bf16
    return forward(x, logits, dequantize_bf16(wgu_q, wgu_s), dequantize_bf16(wd_q, wd_s), k, **kw)


def backward(x, logits, wgu, wd, dout, k, **kw):
    """The layer's gradients for the upstream gradient ``dout`` (float32
    [T, H]) in FP64; see moe_backward.py.  Returns a dict with dx, dlogits,
    dwgu, dwd (and the routing idx, w and dL/dw)."""
    from .moe_backward import backward as f
    return f(x, logits, wgu, wd, dout, k, route, **kw)
