"""Pins for the FP64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the mathematics or a hand derivation
fixes.  ``test_oracle_pins.py`` runs them on the committed oracle and
``test_oracle_mutants.py`` runs them on copies of the oracle with planted
mistakes, each of which must trip at least one pin.

No page prints a worked example, so the pins are: brute force on tiny inputs
(selection by a library sort, the whole layer by a dense every-expert
formulation), closed forms (two-way softmax, identity weights, mean over
experts), special cases that reduce to a textbook routine (k = 1 is a dense
SwiGLU FFN, written with torch's float64 ``F.silu``), invariants (zero input,
exact power-of-two scaling, token and expert relabelling) and the hand-worked
fixture in ``tests/golden/hand_example.json``.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers
def to_bits(a) -> np.ndarray:
    """FP32/FP64 values -> BF16 bit patterns (round to nearest even)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_layer(rng, T, H, I, E, scale_w=True):
    x = to_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    sg = 1 / math.sqrt(H) if scale_w else 1.0
    sd = 1 / math.sqrt(I) if scale_w else 1.0
    wgu = to_bits(rng.standard_normal((E, 2 * I, H)) * sg)
    wd = to_bits(rng.standard_normal((E, H, I)) * sd)
    return x, logits, wgu, wd


def normwise(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


def dense_reference(x, logits, wgu, wd, k):
    """Every expert on every token, then a mask: the brute-force formulation.

    Selection is a library stable sort of -logit (ties keep the lower index);
    weights are a softmax over all E logits, masked to the chosen k and
    renormalised -- algebraically the softmax over the chosen k.
    """
    X, G, D = from_bits(x), from_bits(wgu), from_bits(wd)
    T, E = logits.shape
    I = G.shape[1] // 2
    gate = np.einsum("eih,th->tei", G[:, :I, :], X)
    up = np.einsum("eih,th->tei", G[:, I:, :], X)
    act = gate / (1.0 + np.exp(-gate)) * up
    Y = np.einsum("ehi,tei->teh", D, act)
    L = logits.astype(np.float64)
    order = np.argsort(-L, axis=1, kind="stable")[:, :k]
    P = np.exp(L - L.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    M = np.zeros_like(P)
    rows = np.arange(T)[:, None]
    M[rows, order] = P[rows, order]
    M /= M.sum(axis=1, keepdims=True)
    return np.einsum("te,teh->th", M, Y), order


# ---------------------------------------------------------------- pins
def pin_selection_library_sort(orc):
    """Selection equals a stable library sort by (-logit, index), on tiny
    inputs drawn from a 4-value set so that ties are everywhere."""
    rng = np.random.default_rng(1)
    for E in range(1, 8):
        for k in range(1, E + 1):
            L = rng.choice(np.float32([-1.0, 0.0, 0.5, 1.0]), size=(24, E))
            idx, _ = orc.route(L, k)
            for t in range(L.shape[0]):
                want = sorted(range(E), key=lambda e: (-float(L[t, e]), e))[:k]
                assert list(idx[t]) == want, (E, k, L[t], idx[t], want)


def pin_selection_dominance(orc):
    """Brute force over every ordered k-tuple: the answer is the one tuple
    whose members each beat every later member and every unchosen expert
    (beat = larger logit, or equal logit and smaller index)."""
    rng = np.random.default_rng(2)

    def beats(L, a, b):
        return L[a] > L[b] or (L[a] == L[b] and a < b)

    for E in range(1, 6):
        for k in range(1, E + 1):
            L = rng.choice(np.float32([-0.5, 0.0, 2.0]), size=(8, E))
            idx, _ = orc.route(L, k)
            for t in range(8):
                good = [p for p in itertools.permutations(range(E), k)
                        if all(beats(L[t], p[i], q) for i in range(k)
                               for q in list(p[i + 1:]) + [e for e in range(E) if e not in p])]
                assert len(good) == 1 and list(idx[t]) == list(good[0]), (L[t], idx[t], good)


def pin_signed_zero_tie(orc):
    """-0.0 and +0.0 are equal logits, so the lower index goes first."""
    L = np.float32([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]])
    idx, w = orc.route(L, 2)
    assert idx.tolist() == [[0, 1], [0, 1]]
    assert np.all(w == 0.5)


def pin_weights_closed_form(orc):
    """k = 2: w0 = 1/(1+exp(b-a)) (the logistic function); sum to 1; equal
    logits give exactly 1/2; k = E with equal logits and E = 2^n gives 2^-n."""
    rng = np.random.default_rng(3)
    L = rng.standard_normal((64, 5)).astype(np.float32)
    idx, w = orc.route(L, 2)
    for t in range(64):
        a, b = float(L[t, idx[t, 0]]), float(L[t, idx[t, 1]])
        assert abs(w[t, 0] - 1.0 / (1.0 + math.exp(b - a))) < 1e-15
    for k in (1, 3, 5):
        _, w = orc.route(L, k)
        assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-15)
        assert np.all(np.diff(w, axis=1) <= 0), "slot weights must be non-increasing"
    _, w = orc.route(np.zeros((3, 8), np.float32), 8)
    assert np.all(w == 0.125)


def pin_dense_bruteforce(orc):
    """The whole layer against the dense every-expert formulation, on tiny
    random layers (including ties in the logits) and on the tiny workload's
    shape (T=4, H=256, I=128, E=8, k=2)."""
    rng = np.random.default_rng(4)
    shapes = [(3, 4, 3, 3, 2), (5, 6, 5, 4, 1), (4, 8, 2, 5, 5), (2, 3, 7, 6, 3),
              (4, 256, 128, 8, 2)]
    for (T, H, I, E, k) in shapes:
        x, L, wgu, wd = rand_layer(rng, T, H, I, E)
        if E > 2:
            L[:, 1] = L[:, 2]          # a tie in every token
        out, idx, w = orc.forward(x, L, wgu, wd, k, nthreads=2)
        ref, order = dense_reference(x, L, wgu, wd, k)
        assert np.array_equal(idx, order), (idx, order)
        assert normwise(out, ref) < 1e-13, normwise(out, ref)


def pin_identity_weights(orc):
    """H = I, gate = up = W_down = identity in every expert: every expert
    returns silu(x)*x, so the layer does too, for any routing."""
    rng = np.random.default_rng(5)
    H = 16
    eye = np.eye(H)
    wgu = to_bits(np.stack([np.concatenate([eye, eye])] * 4))
    wd = to_bits(np.stack([eye] * 4))
    xf = rng.standard_normal((6, H))
    x = to_bits(xf)
    X = from_bits(x)
    L = rng.standard_normal((6, 4)).astype(np.float32)
    out, _, _ = orc.forward(x, L, wgu, wd, 3, nthreads=1)
    want = np.vectorize(lambda v: v / (1.0 + math.exp(-v)) * v)(X)
    assert np.max(np.abs(out - want)) <= 1e-15 * max(1.0, np.max(np.abs(want))), \
        np.max(np.abs(out - want))


def pin_mean_over_experts(orc):
    """k = E with equal logits and E = 4: out = mean over experts.  Expert e
    has gate = c_e * identity, up = W_down = identity, so its output is
    silu(c_e x) * x in closed form."""
    rng = np.random.default_rng(6)
    H, E = 8, 4
    cs = [0.5, 1.0, 2.0, -1.0]
    eye = np.eye(H)
    wgu = to_bits(np.stack([np.concatenate([c * eye, eye]) for c in cs]))
    wd = to_bits(np.stack([eye] * E))
    x = to_bits(rng.standard_normal((5, H)))
    X = from_bits(x)
    out, idx, w = orc.forward(x, np.zeros((5, E), np.float32), wgu, wd, E, nthreads=1)
    assert np.all(w == 0.25) and idx.tolist() == [[0, 1, 2, 3]] * 5
    want = np.zeros_like(X)
    for c in cs:
        want += np.vectorize(lambda v: (c * v) / (1.0 + math.exp(-c * v)) * v)(X) / E
    assert np.max(np.abs(out - want)) <= 1e-14, np.max(np.abs(out - want))


def pin_zero_input(orc):
    """x = 0 gives exactly 0 whatever the weights and routing."""
    rng = np.random.default_rng(7)
    _, L, wgu, wd = rand_layer(rng, 3, 64, 32, 6)
    out, _, _ = orc.forward(np.zeros((3, 64), np.uint16), L, wgu, wd, 3)
    assert np.all(out == 0.0)


def pin_k1_textbook(orc):
    """k = 1: the layer is one dense SwiGLU FFN (W_down (silu(W_g x) * W_u x))
    of the top expert with weight 1, written here with torch float64."""
    rng = np.random.default_rng(8)
    T, H, I, E = 5, 24, 12, 4
    x, L, wgu, wd = rand_layer(rng, T, H, I, E)
    out, idx, w = orc.forward(x, L, wgu, wd, 1, nthreads=1)
    assert np.all(w == 1.0)
    X = torch.from_numpy(from_bits(x))
    G = torch.from_numpy(from_bits(wgu))
    D = torch.from_numpy(from_bits(wd))
    for t in range(T):
        e = int(np.argmax(L[t]))
        assert idx[t, 0] == e
        Wg, Wu, Wdn = G[e, :I], G[e, I:], D[e]
        y = Wdn @ (torch.nn.functional.silu(Wg @ X[t]) * (Wu @ X[t]))
        assert np.max(np.abs(out[t] - y.numpy())) < 1e-13


def pin_down_scaling_exact(orc):
    """Doubling W_down (exact in BF16) doubles the output exactly."""
    rng = np.random.default_rng(9)
    x, L, wgu, wd = rand_layer(rng, 4, 32, 16, 5)
    out1, _, _ = orc.forward(x, L, wgu, wd, 2)
    out2, _, _ = orc.forward(x, L, wgu, to_bits(from_bits(wd) * 2.0), 2)
    assert np.array_equal(out2, 2.0 * out1)


def pin_relabelling(orc):
    """Permuting tokens permutes the output rows; permuting expert ids (logit
    columns together with the weight blocks) leaves the output unchanged.
    The expert map (handing over only some experts) changes nothing."""
    rng = np.random.default_rng(10)
    T, H, I, E, k = 6, 32, 16, 7, 3
    x, L, wgu, wd = rand_layer(rng, T, H, I, E)
    out, idx, _ = orc.forward(x, L, wgu, wd, k)
    p = rng.permutation(T)
    outp, _, _ = orc.forward(x[p], L[p], wgu, wd, k)
    assert np.array_equal(outp, out[p])
    q = rng.permutation(E)
    oute, idxe, _ = orc.forward(x, L[:, q], wgu[q], wd[q], k)
    assert np.array_equal(oute, out)
    assert np.array_equal(q[idxe], idx)
    used = np.unique(idx)
    emap = -np.ones(E, np.int32)
    emap[used] = np.arange(len(used))
    outm, _, _ = orc.forward(x, L, wgu[used], wd[used], k, expert_map=emap)
    assert np.array_equal(outm, out)


def pin_hand_example(orc):
    """The hand-worked fixture tests/golden/hand_example.json."""
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    env = {"s1": 1 / (1 + math.exp(-1)), "sm2": -2 / (1 + math.exp(2)),
           "s05": 0.5 / (1 + math.exp(-0.5)), "w0": 1 / (1 + math.exp(-2))}

    def ev(s):
        return eval(s, {"__builtins__": {}}, env)  # expressions from the fixture

    out, idx, w = orc.forward(to_bits(g["x"]), np.float32(g["logits"]),
                              to_bits(g["w_gate_up"]), to_bits(g["w_down"]),
                              g["k"], nthreads=1)
    assert idx.tolist() == g["expected_idx"]
    want_w = np.array([[ev(s) for s in r] for r in g["expected_w"]])
    want = np.array([[ev(s) for s in r] for r in g["expected_out"]])
    assert np.max(np.abs(w - want_w)) < 1e-15
    assert np.max(np.abs(out - want)) < 1e-15, (out, want)


def pin_expert_ffn_matches_layer(orc):
    """The single-expert entry equals the layer with k = 1 and that expert
    forced (its logit made the largest)."""
    rng = np.random.default_rng(11)
    x, L, wgu, wd = rand_layer(rng, 1, 40, 24, 3)
    L[0] = np.float32([0.0, 5.0, -1.0])
    out, _, _ = orc.forward(x, L, wgu, wd, 1)
    y = orc.expert_ffn(x[0], wgu[1], wd[1])
    assert np.array_equal(out[0], y)


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_")]
