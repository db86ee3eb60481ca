"""Pins for the FP64 backward oracle (oracle/moe_backward.py): checks against
things other than the oracle itself.

Each ``pin_*`` function takes a backward function with the signature of
``oracle.backward`` and raises AssertionError when it disagrees with what
the mathematics fixes.  ``test_backward_oracle.py`` runs them on the
committed oracle and on copies of it with planted mistakes, each of which
must trip at least one pin.

The pages print no worked example of the backward pass, so the pins are:
  * torch's float64 autograd (a library's derivative) of the dense
    every-expert formulation of the forward layer, masked by the routing
    weights, on tiny layers (including tied logits);
  * central finite differences of that dense forward, written here in numpy
    and itself tied to the C forward oracle on BF16 inputs;
  * invariants: the softmax gradient sums to zero over the selected experts
    and vanishes elsewhere, untouched experts get zero weight gradients,
    one selected expert gives zero logit gradients, dout = 0 gives zeros and
    doubling dout doubles every gradient exactly;
  * a closed form: identity weights make every expert silu(x) * x, whose
    derivative 2 x sigmoid(x) + x^2 sigmoid(x) (1 - sigmoid(x)) is the
    textbook one.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from tests.oracle_pins import from_bits, normwise, rand_layer, to_bits


def rand_dout(rng, T, H):
    return rng.standard_normal((T, H)).astype(np.float32)


def torch_dense_grads(x, logits, wgu, wd, dout, k):
    """Gradients of sum(out * dout) by torch autograd (float64) on the dense
    formulation: every expert on every token; the selection by a library
    stable sort of -logit; the weights a softmax of the selected logits,
    scattered into an [T, E] mask."""
    X = torch.tensor(from_bits(x), requires_grad=True)
    L = torch.tensor(logits.astype(np.float64), requires_grad=True)
    G = torch.tensor(from_bits(wgu), requires_grad=True)
    D = torch.tensor(from_bits(wd), requires_grad=True)
    dO = torch.tensor(dout.astype(np.float64))
    T, E = logits.shape
    I = G.shape[1] // 2
    order = torch.as_tensor(np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k])
    wsel = torch.softmax(torch.gather(L, 1, order), dim=1)
    M = torch.zeros((T, E), dtype=torch.float64).scatter(1, order, wsel)
    gate = torch.einsum("eih,th->tei", G[:, :I], X)
    up = torch.einsum("eih,th->tei", G[:, I:], X)
    act = torch.nn.functional.silu(gate) * up
    Y = torch.einsum("ehi,tei->teh", D, act)
    out = torch.einsum("te,teh->th", M, Y)
    (out * dO).sum().backward()
    return {"dx": X.grad.numpy(), "dlogits": L.grad.numpy(), "dwgu": G.grad.numpy(), "dwd": D.grad.numpy()}


def dense_forward_f64(X, L, G, D, k, order=None):
    """The dense forward layer on float64 values (numpy); the selection is
    taken from ``order`` when given (so a perturbation cannot change it)."""
    T, E = L.shape
    I = G.shape[1] // 2
    if order is None:
        order = np.argsort(-L, axis=1, kind="stable")[:, :k]
    rows = np.arange(T)[:, None]
    sel = L[rows, order]
    p = np.exp(sel - sel.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    M = np.zeros((T, E))
    M[rows, order] = p
    gate = np.einsum("eih,th->tei", G[:, :I], X)
    up = np.einsum("eih,th->tei", G[:, I:], X)
    act = gate / (1.0 + np.exp(-gate)) * up
    Y = np.einsum("ehi,tei->teh", D, act)
    return np.einsum("te,teh->th", M, Y)


# ---------------------------------------------------------------- pins
def pin_bwd_torch_autograd(backward):
    """Every gradient against torch float64 autograd of the dense
    formulation, on tiny layers and on the tiny workload's shape."""
    rng = np.random.default_rng(21)
    shapes = [(3, 4, 3, 3, 2), (5, 6, 5, 4, 1), (4, 8, 2, 5, 5), (2, 3, 7, 6, 3), (4, 64, 32, 8, 2)]
    for (T, H, I, E, k) in shapes:
        x, L, wgu, wd = rand_layer(rng, T, H, I, E)
        if E > 2:
            L[:, 1] = L[:, 2]          # a tie in every token
        dout = rand_dout(rng, T, H)
        got = backward(x, L, wgu, wd, dout, k)
        want = torch_dense_grads(x, L, wgu, wd, dout, k)
        for name in ("dx", "dwgu", "dwd"):
            assert normwise(got[name], want[name]) < 1e-12, (name, (T, H, I, E, k), normwise(got[name], want[name]))
        # the logit gradient can be exactly zero (k = 1): compare absolutely
        scale = max(1.0, float(np.max(np.abs(want["dlogits"]))))
        assert np.max(np.abs(got["dlogits"] - want["dlogits"])) < 1e-12 * scale, ("dlogits", (T, H, I, E, k))


def pin_bwd_finite_differences(backward):
    """Directional derivatives: (F(p + eps v) - F(p - eps v)) / (2 eps) for
    F = sum(out * dout) of the numpy dense forward, against <grad, v>, for a
    random direction v in each input.  The dense forward is first tied to
    the C forward oracle on the same BF16 inputs."""
    rng = np.random.default_rng(22)
    for (T, H, I, E, k) in [(3, 8, 4, 5, 2), (2, 6, 6, 3, 3)]:
        x, L, wgu, wd = rand_layer(rng, T, H, I, E)
        dout = rand_dout(rng, T, H)
        X, G, D = from_bits(x), from_bits(wgu), from_bits(wd)
        Lf = L.astype(np.float64)
        out_c, idx, _ = oracle.forward(x, L, wgu, wd, k, nthreads=1)
        assert normwise(dense_forward_f64(X, Lf, G, D, k), out_c) < 1e-13
        got = backward(x, L, wgu, wd, dout, k)
        dO = dout.astype(np.float64)

        def F(Xv, Lv, Gv, Dv):
            return float(np.sum(dense_forward_f64(Xv, Lv, Gv, Dv, k, order=idx) * dO))

        eps = 1e-5
        base = [X, Lf, G, D]
        for n, name in enumerate(("dx", "dlogits", "dwgu", "dwd")):
            v = rng.standard_normal(base[n].shape)
            plus = list(base)
            minus = list(base)
            plus[n] = base[n] + eps * v
            minus[n] = base[n] - eps * v
            fd = (F(*plus) - F(*minus)) / (2 * eps)
            an = float(np.sum(got[name] * v))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def pin_bwd_invariants(backward):
    """Structure that holds for any layer: the logit gradient sums to zero
    over each token's selected experts and is zero elsewhere; experts no
    token selects get zero weight gradients; k = 1 gives zero logit
    gradients; dout = 0 gives zeros; 2 dout gives exactly twice every
    gradient (a power of two scales exactly)."""
    rng = np.random.default_rng(23)
    T, H, I, E, k = 4, 16, 8, 9, 3
    x, L, wgu, wd = rand_layer(rng, T, H, I, E)
    dout = rand_dout(rng, T, H)
    got = backward(x, L, wgu, wd, dout, k)
    idx = got["idx"]
    rows = np.arange(T)[:, None]
    sel = got["dlogits"][rows, idx]
    assert np.all(np.abs(sel.sum(axis=1)) <= 1e-15 * np.abs(sel).sum(axis=1).clip(1e-300))
    mask = np.zeros((T, E), bool)
    mask[rows, idx] = True
    assert np.all(got["dlogits"][~mask] == 0.0)
    assert np.any(got["dlogits"][mask] != 0.0)
    untouched = sorted(set(range(E)) - set(idx.ravel().tolist()))
    assert untouched, "the case must leave an expert untouched"
    for e in untouched:
        assert np.all(got["dwgu"][e] == 0.0) and np.all(got["dwd"][e] == 0.0)
    for e in set(idx.ravel().tolist()):
        assert np.any(got["dwgu"][e] != 0.0) and np.any(got["dwd"][e] != 0.0)
    one = backward(x, L, wgu, wd, dout, 1)
    assert np.all(one["dlogits"] == 0.0)
    zero = backward(x, L, wgu, wd, np.zeros_like(dout), k)
    for name in ("dx", "dlogits", "dwgu", "dwd"):
        assert np.all(zero[name] == 0.0), name
    two = backward(x, L, wgu, wd, 2 * dout, k)
    for name in ("dx", "dlogits", "dwgu", "dwd"):
        assert np.array_equal(two[name], 2 * got[name]), name


def pin_bwd_identity_closed_form(backward):
    """H = I and gate = up = W_down = identity in every expert: each expert
    maps x to silu(x) * x = x^2 sigmoid(x), so for any routing
    dx = dout * (2 x s + x^2 s (1 - s)) with s = sigmoid(x), the logit
    gradient vanishes (every selected expert returns the same vector) and
    dW_down[e] = sum over e's tokens of w * dout (x) a."""
    rng = np.random.default_rng(24)
    H, E, T, k = 12, 4, 5, 2
    eye = np.eye(H)
    wgu = to_bits(np.stack([np.concatenate([eye, eye])] * E))
    wd = to_bits(np.stack([eye] * E))
    x = to_bits(rng.standard_normal((T, H)))
    X = from_bits(x)
    L = rng.standard_normal((T, E)).astype(np.float32)
    dout = rand_dout(rng, T, H)
    dO = dout.astype(np.float64)
    got = backward(x, L, wgu, wd, dout, k)
    s = 1.0 / (1.0 + np.exp(-X))
    want_dx = dO * (2 * X * s + X * X * s * (1 - s))
    assert np.max(np.abs(got["dx"] - want_dx)) <= 1e-14 * max(1.0, np.max(np.abs(want_dx)))
    assert np.max(np.abs(got["dlogits"])) <= 1e-14 * max(1.0, np.max(np.abs(dO)) * np.max(X * X))
    a = X * X * s
    for e in range(E):
        want = np.zeros((H, H))
        for t in range(T):
            for j in range(k):
                if got["idx"][t, j] == e:
                    want += got["w"][t, j] * np.outer(dO[t], a[t])
        assert np.max(np.abs(got["dwd"][e] - want)) <= 1e-14 * max(1.0, np.max(np.abs(want)))
    assert math.isfinite(float(np.sum(got["dwgu"])))


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_")]
