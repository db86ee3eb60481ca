"""FP64 oracle for the backward pass of the routed MoE SwiGLU FFN.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): the product never
imports it and it imports nothing of the product.

What it computes.  The Mixture-of-Kittens article ("커서가 MoE 학습 메가커널
믹스처 오브 키튼스를 아파치 2.0으로 공개했다", section 2.37배는 어떤 기준선과
비교한 숫자인가) measures the MoE layer's forward and backward passes in
training; neither page writes the backward out.  The layer's reading: the
gradients of the forward layer (the definition in ``moe_oracle.c``) with
respect to its four inputs, for an upstream gradient dout = dL/dout [T, H]
(FP32), by the chain rule, every intermediate in FP64:

  per token t and slot j, expert e = s_j, routing weight w = w_j:
    g = W_gate[e] x_t,  u = W_up[e] x_t,  s = sigmoid(g),  a = g s u
    q = W_down[e]^T dout_t                      (dL/dy_j = w dout_t)
    dw_j = a . q                                 (dL/dw_j = dout_t . y_j)
    da = w q
    dg = da u s (1 + g (1 - s))                  (d(g sigmoid(g))/dg)
    du = da g s
    dx_t         += W_gate[e]^T dg + W_up[e]^T du
    dW_down[e]   += (w dout_t) a^T
    dW_gate[e]   += dg x_t^T,   dW_up[e] += du x_t^T
  and for the router logits, the softmax over the k selected logits:
    dlogits[t, s_j] = w_j (dw_j - sum_m w_m dw_m),  0 for every other expert.

The top-k selection is piecewise constant in the logits, so the unselected
experts' logits get zero gradient (the plain reading: the derivative where it
exists).  Experts that no token selects get zero weight gradients.

How.  For each expert, the rows of its assignments are gathered (tokens in
ascending order; the order does not matter in FP64 beyond rounding) and each
line above is one numpy FP64 expression or matmul; nothing is blocked, fused
or reordered beyond that.  BF16 inputs convert to FP64 exactly, FP32 inputs
too.  The selection and the weights come from the forward oracle's routing.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> their exact values as float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sigmoid(v: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-v))


def expert_backward(xe, de, we, wgu_e, wd_e):
    """One expert's part of the backward pass, for the n assignments routed
    to it: xe [n, H] and de [n, H] the tokens' x and dout rows (float64),
    we [n] their routing weights, wgu_e uint16 [2I, H] and wd_e uint16
    [H, I] its BF16 weights.  Returns (dx rows [n, H] -- this expert's
    contribution to each token's dx --, dw [n] = dL/dw, dW_gate_up [2I, H],
    dW_down [H, I]), all float64."""
    I = wgu_e.shape[0] // 2
    Wg = bf16_to_f64(wgu_e[:I])                 # [I, H]
    Wu = bf16_to_f64(wgu_e[I:])
    Wd = bf16_to_f64(wd_e)                      # [H, I]
    g = xe @ Wg.T
    u = xe @ Wu.T
    s = sigmoid(g)
    a = g * s * u
    q = de @ Wd                                 # rows: W_down^T dout_t
    dw = np.sum(a * q, axis=1)
    da = we[:, None] * q
    dg = da * u * s * (1.0 + g * (1.0 - s))
    du = da * g * s
    dx_rows = dg @ Wg + du @ Wu
    dwd = (we[:, None] * de).T @ a
    dwgu = np.concatenate([dg.T @ xe, du.T @ xe])
    return dx_rows, dw, dwgu, dwd


def backward(x, logits, wgu, wd, dout, k, route, *, expert_map=None):
    """The layer's gradients in FP64.

    x uint16 [T, H] (BF16 bits); logits float32 [T, E]; wgu uint16
    [Eb, 2I, H]; wd uint16 [Eb, H, I]; dout float32 [T, H]; ``route`` the
    forward oracle's routing, (logits, k) -> (idx int32 [T, k], w float64
    [T, k]).  With ``expert_map`` (int32 [E], -1 = absent) the weight arrays
    hold only the blocks the map names (every selected expert must be
    present), and so do the returned weight gradients.

    Returns a dict: dx [T, H], dlogits [T, E], dwgu [Eb, 2I, H], dwd
    [Eb, H, I] (float64), and idx, w, dw (the routing and dL/dw [T, k]).
    """
    xf = bf16_to_f64(x)
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    douf = np.ascontiguousarray(dout, dtype=np.float32).astype(np.float64)
    T, H = xf.shape
    E = logits.shape[1]
    Eb, I2, _ = wgu.shape
    I = I2 // 2
    assert wgu.shape == (Eb, 2 * I, H) and wd.shape == (Eb, H, I) and douf.shape == (T, H)
    if expert_map is None:
        assert Eb == E
        expert_map = np.arange(E, dtype=np.int32)
    idx, w = route(logits, k)

    dx = np.zeros((T, H))
    dwgu = np.zeros((Eb, 2 * I, H))
    dwd = np.zeros((Eb, H, I))
    dw = np.zeros((T, k))
    for e in np.unique(idx):
        b = int(expert_map[e])
        if b < 0:
            raise ValueError(f"expert {e} is selected but has no weights")
        tok, slot = np.nonzero(idx == e)          # ascending token order
        dx_rows, dw_e, dwgu[b], dwd[b] = expert_backward(xf[tok], douf[tok], w[tok, slot], wgu[b], wd[b])
        dx[tok] += dx_rows                        # a token picks e at most once
        dw[tok, slot] = dw_e

    dlogits = np.zeros((T, E))
    S = np.sum(w * dw, axis=1)
    rows = np.arange(T)[:, None]
    dlogits[rows, idx] = w * (dw - S[:, None])
    return {"dx": dx, "dlogits": dlogits, "dwgu": dwgu, "dwd": dwd, "idx": idx, "w": w, "dw": dw}
