"""ctypes binding of libmoeffn.so (C ABI in include/moe_ffn.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C names and take torch tensors for device
buffers; the stream defaults to torch's current stream.  There is no CPU
fallback: if the library is not built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_CUDA = 3
MOE_ERR_NO_MEMORY = 4
MOE_ERR_WORKSPACE_TOO_SMALL = 5
MOE_ERR_TIMEOUT = 6

MOE_PATH_AUTO = 0
MOE_PATH_DECODE = 1
MOE_PATH_GROUPED = 2
MOE_PATH_DECODE_FUSED = 3  # reported only: the decode path for T <= 4 as one kernel
MOE_PATH_BACKWARD = 4      # reported only: moe_ffn_backward's kernels
MOE_PATH_TRAIN_FORWARD = 5   # reported only: moe_ffn_forward_train
MOE_PATH_TRAIN_BACKWARD = 6  # reported only: moe_ffn_backward_train
MOE_MAX_STAGES = 12

EXPORTED = ["moe_ffn_forward", "moe_ffn_workspace_bytes", "moe_ffn_forward_ex",
            "moe_ffn_host_workspace_bytes", "moe_ffn_forward_host", "moe_ffn_status_string",
            "moe_ffn_stage_name", "moe_ffn_device_faults", "moe_ffn_forward_noalloc",
            "moe_ffn_router_workspace_bytes", "moe_ffn_forward_router", "moe_ffn_forward_mxfp8",
            "moe_ffn_backward_workspace_bytes", "moe_ffn_backward", "moe_ffn_train_state_bytes",
            "moe_ffn_forward_train", "moe_ffn_backward_train"]

# Size of the library's fixed scratch array used by moe_ffn_forward_noalloc.
MOE_FFN_NOALLOC_SCRATCH_BYTES = 16 << 20
# Leading bytes of a workspace that hold the state kept between calls.
MOE_FFN_WORKSPACE_STATE_BYTES = 16384

# Values moe_ffn_opts.exchange_out receives from a fused decode call.
EXCHANGE_BARRIER = 1
EXCHANGE_TAGGED = 2


class moe_ffn_opts(ctypes.Structure):
    """Mirror of ``struct moe_ffn_opts``."""
    _fields_ = [("path", ctypes.c_int32), ("decode_max_tokens", ctypes.c_int32),
                ("gate_up_warps", ctypes.c_int32), ("down_warps", ctypes.c_int32),
                ("gemm_ctas", ctypes.c_int32), ("test_wait_limit_us", ctypes.c_int32),
                ("test_skip_arrival", ctypes.c_int32), ("reserved_in", ctypes.c_int32 * 1),
                ("stage_events", ctypes.c_void_p), ("exchange_out", ctypes.c_void_p),
                ("n_stages", ctypes.c_int32), ("path_taken", ctypes.c_int32),
                ("reserved_out", ctypes.c_int32 * 2)]


class MoeFfnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {moe_ffn_status_string(status)} (status {status})")


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    """The library this process loads: MOE_FFN_LIB if set (e.g. the
    instrumented timeline build), else the in-tree build."""
    return os.environ.get("MOE_FFN_LIB") or _build.LIB


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.moe_ffn_forward.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp]
            L.moe_ffn_workspace_bytes.argtypes = [i64] * 5
            L.moe_ffn_workspace_bytes.restype = ctypes.c_size_t
            L.moe_ffn_forward_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp,
                                             ctypes.c_size_t, vp, vp,
                                             ctypes.POINTER(moe_ffn_opts), vp]
            L.moe_ffn_host_workspace_bytes.argtypes = [i64] * 5
            L.moe_ffn_host_workspace_bytes.restype = ctypes.c_size_t
            L.moe_ffn_forward_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp,
                                               ctypes.c_size_t, ctypes.POINTER(moe_ffn_opts), vp]
            L.moe_ffn_status_string.argtypes = [i32]
            L.moe_ffn_status_string.restype = ctypes.c_char_p
            L.moe_ffn_stage_name.argtypes = [i32, i32]
            L.moe_ffn_stage_name.restype = ctypes.c_char_p
            L.moe_ffn_device_faults.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
            L.moe_ffn_forward_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp]
            L.moe_ffn_router_workspace_bytes.argtypes = [i64] * 5
            L.moe_ffn_router_workspace_bytes.restype = ctypes.c_size_t
            L.moe_ffn_forward_router.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp,
                                                 ctypes.c_size_t, vp, vp, vp,
                                                 ctypes.POINTER(moe_ffn_opts), vp]
            L.moe_ffn_forward_mxfp8.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp,
                                                ctypes.c_size_t, vp, vp, ctypes.POINTER(moe_ffn_opts), vp]
            L.moe_ffn_backward_workspace_bytes.argtypes = [i64] * 5
            L.moe_ffn_backward_workspace_bytes.restype = ctypes.c_size_t
            L.moe_ffn_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                                           ctypes.c_size_t, ctypes.POINTER(moe_ffn_opts), vp]
            L.moe_ffn_train_state_bytes.argtypes = [i64] * 5
            L.moe_ffn_train_state_bytes.restype = ctypes.c_size_t
            L.moe_ffn_forward_train.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, ctypes.c_size_t,
                                                ctypes.POINTER(moe_ffn_opts), vp]
            L.moe_ffn_backward_train.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                                                 ctypes.c_size_t, ctypes.POINTER(moe_ffn_opts), vp]
            for f in (L.moe_ffn_forward, L.moe_ffn_forward_ex, L.moe_ffn_forward_host,
                      L.moe_ffn_device_faults, L.moe_ffn_forward_noalloc, L.moe_ffn_forward_router,
                      L.moe_ffn_forward_mxfp8, L.moe_ffn_backward, L.moe_ffn_forward_train,
                      L.moe_ffn_backward_train):
                f.restype = i32
            if hasattr(L, "moe_ffn_debug_fused_timeline"):   # instrumented build only
                L.moe_ffn_debug_fused_timeline.argtypes = [vp, i32]
                L.moe_ffn_debug_fused_timeline.restype = i32
            _lib = L
    return _lib


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status, what):
    if status != MOE_OK:
        raise MoeFfnError(status, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _shape(x, logits, w_gate_up, w_down):
    T, H = x.shape
    E = logits.shape[1]
    I = w_down.shape[2]
    if logits.shape[0] != T or tuple(w_gate_up.shape) != (E, 2 * I, H) or tuple(w_down.shape) != (E, H, I):
        raise ValueError(f"shape mismatch: x {tuple(x.shape)} logits {tuple(logits.shape)} "
                         f"w_gate_up {tuple(w_gate_up.shape)} w_down {tuple(w_down.shape)}")
    return T, H, I, E


def _dev(t, dtype, name):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def moe_ffn_status_string(status: int) -> str:
    return lib().moe_ffn_status_string(int(status)).decode()


def moe_ffn_stage_name(path: int, stage: int):
    r = lib().moe_ffn_stage_name(int(path), int(stage))
    return None if r is None else r.decode()


def moe_ffn_workspace_bytes(T, H, I, E, k) -> int:
    return int(lib().moe_ffn_workspace_bytes(T, H, I, E, k))


def moe_ffn_host_workspace_bytes(T, H, I, E, k) -> int:
    return int(lib().moe_ffn_host_workspace_bytes(T, H, I, E, k))


def moe_ffn_device_faults(clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().moe_ffn_device_faults(ctypes.byref(v), int(clear)), "moe_ffn_device_faults")
    return int(v.value)


def moe_ffn_forward(x, logits, w_gate_up, w_down, k: int, out=None, stream=None):
    """out[T,H] f32 = layer(x bf16 [T,H], logits f32 [T,E], weights).

    Uses a stream-ordered temporary workspace inside the library.
    """
    T, H, I, E = _shape(x, logits, w_gate_up, w_down)
    for t, d, n in ((x, torch.bfloat16, "x"), (logits, torch.float32, "logits"),
                    (w_gate_up, torch.bfloat16, "w_gate_up"), (w_down, torch.bfloat16, "w_down")):
        _dev(t, d, n)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(lib().moe_ffn_forward(_ptr(x), _ptr(logits), _ptr(w_gate_up), _ptr(w_down),
                                 T, H, I, E, k, _ptr(out), _stream(stream)), "moe_ffn_forward")
    return out


def moe_ffn_forward_noalloc(x, logits, w_gate_up, w_down, k: int, out=None, stream=None):
    """The forward pass for callers that cannot allocate device memory: the
    library keeps its scratch in a fixed device array of
    MOE_FFN_NOALLOC_SCRATCH_BYTES, shared by every call (order calls on one
    stream).  ``out`` should be passed by such callers; when it is None this
    wrapper allocates it with torch, for convenience only."""
    T, H, I, E = _shape(x, logits, w_gate_up, w_down)
    for t, d, n in ((x, torch.bfloat16, "x"), (logits, torch.float32, "logits"),
                    (w_gate_up, torch.bfloat16, "w_gate_up"), (w_down, torch.bfloat16, "w_down")):
        _dev(t, d, n)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    _check(lib().moe_ffn_forward_noalloc(_ptr(x), _ptr(logits), _ptr(w_gate_up), _ptr(w_down),
                                         T, H, I, E, k, _ptr(out), _stream(stream)),
           "moe_ffn_forward_noalloc")
    return out


def new_workspace(T, H, I, E, k, device="cuda", host=False):
    """A workspace tensor big enough for this shape (256-byte aligned).

    Its state bytes are zeroed: torch's caching allocator may hand out
    memory that served as another workspace and then held other data."""
    n = (moe_ffn_host_workspace_bytes if host else moe_ffn_workspace_bytes)(T, H, I, E, k)
    if n == 0:
        raise MoeFfnError(MOE_ERR_UNSUPPORTED_SHAPE, "workspace size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:MOE_FFN_WORKSPACE_STATE_BYTES].zero_()
    return ws


def moe_ffn_forward_ex(x, logits, w_gate_up, w_down, k: int, out=None, workspace=None,
                       topk_idx=None, topk_w=None, opts: moe_ffn_opts | None = None,
                       stream=None):
    """The forward pass with a caller-owned workspace, optional routing
    outputs (int32 / float32 [T,k]) and options.  Returns out."""
    T, H, I, E = _shape(x, logits, w_gate_up, w_down)
    for t, d, n in ((x, torch.bfloat16, "x"), (logits, torch.float32, "logits"),
                    (w_gate_up, torch.bfloat16, "w_gate_up"), (w_down, torch.bfloat16, "w_down")):
        _dev(t, d, n)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = new_workspace(T, H, I, E, k, device=x.device)
    if topk_idx is not None:
        _dev(topk_idx, torch.int32, "topk_idx")
    if topk_w is not None:
        _dev(topk_w, torch.float32, "topk_w")
    _check(lib().moe_ffn_forward_ex(
        _ptr(x), _ptr(logits), _ptr(w_gate_up), _ptr(w_down), T, H, I, E, k, _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(topk_idx),
        _ptr(topk_w), ctypes.byref(opts) if opts is not None else None, _stream(stream)),
        "moe_ffn_forward_ex")
    return out


def moe_ffn_router_workspace_bytes(T, H, I, E, k) -> int:
    return int(lib().moe_ffn_router_workspace_bytes(T, H, I, E, k))


def new_router_workspace(T, H, I, E, k, device="cuda"):
    """A workspace for moe_ffn_forward_router (state bytes zeroed)."""
    n = moe_ffn_router_workspace_bytes(T, H, I, E, k)
    if n == 0:
        raise MoeFfnError(MOE_ERR_UNSUPPORTED_SHAPE, "workspace size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:MOE_FFN_WORKSPACE_STATE_BYTES].zero_()
    return ws


def moe_ffn_forward_router(x, w_router, router_bias, w_gate_up, w_down, k: int, out=None,
                           workspace=None, logits=None, topk_idx=None, topk_w=None,
                           opts: moe_ffn_opts | None = None, stream=None):
    """The layer with its router projection inside the call: x bf16 [T,H],
    w_router bf16 [E,H], router_bias f32 [E] or None; optional outputs
    logits f32 [T,E], topk_idx int32 / topk_w f32 [T,k].  Returns out."""
    T, H = x.shape
    E = w_router.shape[0]
    I = w_down.shape[2]
    if tuple(w_router.shape) != (E, H) or tuple(w_gate_up.shape) != (E, 2 * I, H) \
            or tuple(w_down.shape) != (E, H, I):
        raise ValueError("shape mismatch")
    for t, d, n in ((x, torch.bfloat16, "x"), (w_router, torch.bfloat16, "w_router"),
                    (w_gate_up, torch.bfloat16, "w_gate_up"), (w_down, torch.bfloat16, "w_down")):
        _dev(t, d, n)
    if router_bias is not None:
        _dev(router_bias, torch.float32, "router_bias")
    for t, d, n in ((logits, torch.float32, "logits"), (topk_idx, torch.int32, "topk_idx"),
                    (topk_w, torch.float32, "topk_w")):
        if t is not None:
            _dev(t, d, n)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = new_router_workspace(T, H, I, E, k, device=x.device)
    _check(lib().moe_ffn_forward_router(
        _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w_gate_up), _ptr(w_down), T, H, I, E, k,
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(logits),
        _ptr(topk_idx), _ptr(topk_w), ctypes.byref(opts) if opts is not None else None,
        _stream(stream)), "moe_ffn_forward_router")
    return out


def mx_scale_bytes(K: int) -> int:
    """Bytes per row of an MXFP8 scale array for rows of K elements
    (MOE_FFN_MX_SCALE_BYTES)."""
    return (K // 32 + 15) // 16 * 16


def moe_ffn_forward_mxfp8(x, logits, w_gate_up_q, w_gate_up_s, w_down_q, w_down_s, k: int, out=None,
                          workspace=None, topk_idx=None, topk_w=None, opts: moe_ffn_opts | None = None,
                          stream=None):
    """The layer with MXFP8 expert weights (fused decode kernel up to four
    tokens, tensor-core grouped path beyond; MOE_PATH_DECODE forces the
    general decode kernels, up to 64 tokens): x bf16 [T,H],
    logits f32 [T,E], E4M3 codes uint8 w_gate_up_q [E,2I,H] / w_down_q
    [E,H,I], E8M0 scales uint8 w_gate_up_s [E,2I,mx_scale_bytes(H)] /
    w_down_s [E,H,mx_scale_bytes(I)].  Returns out f32 [T,H]."""
    T, H = x.shape
    E = logits.shape[1]
    I = w_down_q.shape[2]
    if tuple(w_gate_up_q.shape) != (E, 2 * I, H) or tuple(w_down_q.shape) != (E, H, I) \
            or tuple(w_gate_up_s.shape) != (E, 2 * I, mx_scale_bytes(H)) \
            or tuple(w_down_s.shape) != (E, H, mx_scale_bytes(I)):
        raise ValueError("shape mismatch")
    for t, d, n in ((x, torch.bfloat16, "x"), (logits, torch.float32, "logits"),
                    (w_gate_up_q, torch.uint8, "w_gate_up_q"), (w_gate_up_s, torch.uint8, "w_gate_up_s"),
                    (w_down_q, torch.uint8, "w_down_q"), (w_down_s, torch.uint8, "w_down_s")):
        _dev(t, d, n)
    for t, d, n in ((topk_idx, torch.int32, "topk_idx"), (topk_w, torch.float32, "topk_w")):
        if t is not None:
            _dev(t, d, n)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = new_workspace(T, H, I, E, k, device=x.device)
    _check(lib().moe_ffn_forward_mxfp8(
        _ptr(x), _ptr(logits), _ptr(w_gate_up_q), _ptr(w_gate_up_s), _ptr(w_down_q), _ptr(w_down_s),
        T, H, I, E, k, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(topk_idx), _ptr(topk_w), ctypes.byref(opts) if opts is not None else None,
        _stream(stream)), "moe_ffn_forward_mxfp8")
    return out


def moe_ffn_forward_host(x_host, logits_host, w_gate_up, w_down, k: int, out_host,
                         workspace, opts: moe_ffn_opts | None = None, stream=None):
    """End-to-end call: x_host / logits_host / out_host are (pinned) CPU
    tensors; copies in and out are enqueued with the forward pass."""
    T, H = x_host.shape
    E = logits_host.shape[1]
    I = w_down.shape[2]
    for t in (x_host, logits_host, out_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors")
    _check(lib().moe_ffn_forward_host(
        _ptr(x_host), _ptr(logits_host), _ptr(w_gate_up), _ptr(w_down), T, H, I, E, k,
        _ptr(out_host), _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(opts) if opts is not None else None, _stream(stream)),
        "moe_ffn_forward_host")
    return out_host


def moe_ffn_backward_workspace_bytes(T, H, I, E, k) -> int:
    return int(lib().moe_ffn_backward_workspace_bytes(T, H, I, E, k))


def new_backward_workspace(T, H, I, E, k, device="cuda"):
    """A workspace for moe_ffn_backward (state bytes zeroed, so that forward
    calls may share it)."""
    n = moe_ffn_backward_workspace_bytes(T, H, I, E, k)
    if n == 0:
        raise MoeFfnError(MOE_ERR_UNSUPPORTED_SHAPE, "workspace size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:MOE_FFN_WORKSPACE_STATE_BYTES].zero_()
    return ws


def moe_ffn_backward(x, logits, w_gate_up, w_down, dout, k: int, dx=None, dlogits=None, dw_gate_up=None,
                     dw_down=None, workspace=None, opts: moe_ffn_opts | None = None, stream=None):
    """The layer's gradients for dout f32 [T,H]: returns (dx f32 [T,H],
    dlogits f32 [T,E], dw_gate_up f32 [E,2I,H], dw_down f32 [E,H,I]).
    Without ``workspace`` the library allocates one stream-ordered."""
    T, H, I, E = _shape(x, logits, w_gate_up, w_down)
    for t, d, n in ((x, torch.bfloat16, "x"), (logits, torch.float32, "logits"),
                    (w_gate_up, torch.bfloat16, "w_gate_up"), (w_down, torch.bfloat16, "w_down"),
                    (dout, torch.float32, "dout")):
        _dev(t, d, n)
    if tuple(dout.shape) != (T, H):
        raise ValueError(f"dout must be [{T}, {H}], got {tuple(dout.shape)}")
    dev = x.device
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.float32, device=dev)
    if dlogits is None:
        dlogits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if dw_gate_up is None:
        dw_gate_up = torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev)
    if dw_down is None:
        dw_down = torch.empty((E, H, I), dtype=torch.float32, device=dev)
    for t, shape, n in ((dx, (T, H), "dx"), (dlogits, (T, E), "dlogits"), (dw_gate_up, (E, 2 * I, H), "dw_gate_up"),
                        (dw_down, (E, H, I), "dw_down")):
        _dev(t, torch.float32, n)
        if tuple(t.shape) != shape:
            raise ValueError(f"{n} must be {list(shape)}, got {tuple(t.shape)}")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().moe_ffn_backward(
        _ptr(x), _ptr(logits), _ptr(w_gate_up), _ptr(w_down), _ptr(dout), T, H, I, E, k, _ptr(dx),
        _ptr(dlogits), _ptr(dw_gate_up), _ptr(dw_down), _ptr(workspace), nbytes,
        ctypes.byref(opts) if opts is not None else None, _stream(stream)), "moe_ffn_backward")
    return dx, dlogits, dw_gate_up, dw_down


def moe_ffn_train_state_bytes(T, H, I, E, k) -> int:
    return int(lib().moe_ffn_train_state_bytes(T, H, I, E, k))


def new_train_state(T, H, I, E, k, device="cuda"):
    """A state buffer for the training pair (moe_ffn_forward_train, then
    moe_ffn_backward_train)."""
    n = moe_ffn_train_state_bytes(T, H, I, E, k)
    if n == 0:
        raise MoeFfnError(MOE_ERR_UNSUPPORTED_SHAPE, "state size")
    st = torch.empty(n, dtype=torch.uint8, device=device)
    st[:MOE_FFN_WORKSPACE_STATE_BYTES].zero_()
    return st


def moe_ffn_forward_train(x, logits, w_gate_up, w_down, k: int, state, out=None,
                          opts: moe_ffn_opts | None = None, stream=None):
    """The layer's output f32 [T,H], keeping in ``state`` (from
    new_train_state) what moe_ffn_backward_train needs."""
    T, H, I, E = _shape(x, logits, w_gate_up, w_down)
    for t, d, n in ((x, torch.bfloat16, "x"), (logits, torch.float32, "logits"),
                    (w_gate_up, torch.bfloat16, "w_gate_up"), (w_down, torch.bfloat16, "w_down"),
                    (state, torch.uint8, "state")):
        _dev(t, d, n)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _dev(out, torch.float32, "out")
    if tuple(out.shape) != (T, H):
        raise ValueError(f"out must be [{T}, {H}], got {tuple(out.shape)}")
    _check(lib().moe_ffn_forward_train(
        _ptr(x), _ptr(logits), _ptr(w_gate_up), _ptr(w_down), T, H, I, E, k, _ptr(out), _ptr(state),
        state.numel(), ctypes.byref(opts) if opts is not None else None, _stream(stream)), "moe_ffn_forward_train")
    return out


def moe_ffn_backward_train(x, logits, w_gate_up, w_down, dout, k: int, state, dx=None, dlogits=None,
                           dw_gate_up=None, dw_down=None, opts: moe_ffn_opts | None = None, stream=None):
    """The layer's gradients for dout f32 [T,H], reading g and u from the
    state a moe_ffn_forward_train call on the same x, logits and weights
    left: returns (dx, dlogits, dw_gate_up, dw_down) as moe_ffn_backward
    does."""
    T, H, I, E = _shape(x, logits, w_gate_up, w_down)
    for t, d, n in ((x, torch.bfloat16, "x"), (logits, torch.float32, "logits"),
                    (w_gate_up, torch.bfloat16, "w_gate_up"), (w_down, torch.bfloat16, "w_down"),
                    (dout, torch.float32, "dout"), (state, torch.uint8, "state")):
        _dev(t, d, n)
    if tuple(dout.shape) != (T, H):
        raise ValueError(f"dout must be [{T}, {H}], got {tuple(dout.shape)}")
    dev = x.device
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.float32, device=dev)
    if dlogits is None:
        dlogits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if dw_gate_up is None:
        dw_gate_up = torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev)
    if dw_down is None:
        dw_down = torch.empty((E, H, I), dtype=torch.float32, device=dev)
    for t, shape, n in ((dx, (T, H), "dx"), (dlogits, (T, E), "dlogits"), (dw_gate_up, (E, 2 * I, H), "dw_gate_up"),
                        (dw_down, (E, H, I), "dw_down")):
        _dev(t, torch.float32, n)
        if tuple(t.shape) != shape:
            raise ValueError(f"{n} must be {list(shape)}, got {tuple(t.shape)}")
    _check(lib().moe_ffn_backward_train(
        _ptr(x), _ptr(logits), _ptr(w_gate_up), _ptr(w_down), _ptr(dout), T, H, I, E, k, _ptr(dx), _ptr(dlogits),
        _ptr(dw_gate_up), _ptr(dw_down), _ptr(state), state.numel(),
        ctypes.byref(opts) if opts is not None else None, _stream(stream)), "moe_ffn_backward_train")
    return dx, dlogits, dw_gate_up, dw_down


def stage_event_array(events):
    """A C array of cudaEvent_t for moe_ffn_opts.stage_events, from
    MOE_MAX_STAGES + 1 torch.cuda.Event objects that have been recorded once
    (torch creates the underlying event on first record)."""
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return arr
