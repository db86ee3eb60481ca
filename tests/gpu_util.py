"""Helpers for the GPU tests: seeded inputs, the CUDA call through the C ABI,
the oracle on the same bytes, and the acceptance check.

Acceptance (written here once, used by every parity test):
  * routing indices bit-exact against the oracle;
  * routing weights within 2e-6 relative (FP32 expf/divide vs FP64);
  * output: ||y - y_ref||_2 / ||y_ref||_2 <= 1e-4 and
            max |y - y_ref| <= 1e-3 * rms(y_ref).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth

NORMWISE_TOL = 1e-4
MAXABS_RMS_TOL = 1e-3
WEIGHT_RTOL = 2e-6

PATHS = {"decode": m.MOE_PATH_DECODE, "grouped": m.MOE_PATH_GROUPED}


def custom(T, H, I, E, k, bias_var=0.0, name="test_layer"):
    wl = dataclasses.replace(synth.WORKLOADS["tiny_t4_h256_i128_e8_k2"], name=name, T=(T,),
                             H=H, I=I, E=E, k=k, bias_var=bias_var)
    return wl


def make_layer(wl, T, device="cuda", call=0, weights_device="cpu"):
    """(x, logits, wgu, wd) on `device`, weights drawn on weights_device."""
    wgu, wd = synth.make_weights(wl, device=weights_device)
    x, logits = synth.make_tokens(wl, T, call=call)
    return x.to(device), logits.to(device), wgu.to(device), wd.to(device)


def run_gpu(x, logits, wgu, wd, k, path="decode", **opt_fields):
    """The layer through moe_ffn_forward_ex; returns (out, idx, w) on the host."""
    T = x.shape[0]
    idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    o = m.moe_ffn_opts()
    o.path = PATHS[path] if isinstance(path, str) else path
    for f, v in opt_fields.items():
        setattr(o, f, v)
    out = m.moe_ffn_forward_ex(x, logits, wgu, wd, k, topk_idx=idx, topk_w=w, opts=o)
    torch.cuda.synchronize()
    if T:
        want = {m.MOE_PATH_DECODE: (m.MOE_PATH_DECODE, m.MOE_PATH_DECODE_FUSED),
                m.MOE_PATH_GROUPED: (m.MOE_PATH_GROUPED,)}.get(o.path)
        assert want is None or o.path_taken in want, (o.path, o.path_taken)
    return out.cpu(), idx.cpu(), w.cpu()


def oracle_ref(x, logits, wgu, wd, k, tokens=None):
    """The oracle on the exact bytes (optionally only rows `tokens`), handing
    it only the experts those tokens select."""
    if tokens is None:
        tokens = np.arange(x.shape[0])
    tokens = torch.as_tensor(np.asarray(tokens), dtype=torch.long)
    L = logits.detach()[tokens.to(logits.device)].cpu().numpy()
    xb = synth.bf16_bits(x.detach()[tokens.to(x.device)])
    idx, _ = oracle.route(L, k)
    used = np.unique(idx)
    emap = -np.ones(L.shape[1], np.int32)
    emap[used] = np.arange(len(used), dtype=np.int32)
    sel = torch.as_tensor(used, dtype=torch.long, device=wgu.device)
    out, idx, w = oracle.forward(xb, L, synth.bf16_bits(wgu.index_select(0, sel)),
                                 synth.bf16_bits(wd.index_select(0, sel)), k, expert_map=emap)
    return out, idx, w


def errors(out, ref):
    y = out.double().numpy() if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    d = y - ref
    nref = np.linalg.norm(ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return (float(np.linalg.norm(d) / nref) if nref > 0 else float(np.linalg.norm(d)),
            float(np.max(np.abs(d))) if d.size else 0.0, rms)


def assert_accepted(out, idx, w, ref_out, ref_idx, ref_w, what=""):
    assert np.array_equal(idx.numpy(), ref_idx), f"{what}: routing indices differ"
    rel = np.abs(w.double().numpy() - ref_w) / np.maximum(np.abs(ref_w), 1e-30)
    assert rel.max() <= WEIGHT_RTOL, f"{what}: weight rel err {rel.max():.3g}"
    nw, mx, rms = errors(out, ref_out)
    if rms == 0.0:
        assert mx == 0.0, f"{what}: reference is zero but output is not"
        return nw, mx
    assert nw <= NORMWISE_TOL, f"{what}: normwise {nw:.3g} > {NORMWISE_TOL}"
    assert mx <= MAXABS_RMS_TOL * rms, f"{what}: max abs {mx:.3g} > {MAXABS_RMS_TOL}*rms ({rms:.3g})"
    return nw, mx
