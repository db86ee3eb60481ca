"""Pins for the oracle's router projection (oracle/router.py): checks against
closed forms, a library matmul where every sum is exact, exact rational
arithmetic, and the two places where a plain floating-point sum goes wrong
(catastrophic cancellation, double rounding).

Each ``pin_*`` takes the ``router_logits`` function under test and raises
AssertionError when it disagrees; ``test_router_oracle.py`` runs them on the
committed function and on copies with planted mistakes.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from tests.oracle_pins import from_bits, to_bits


def _exact_f32(values) -> np.float32:
    """Round the exact rational sum of ``values`` to float32 by hand (ties to
    even), without floating-point summation."""
    s = sum((Fraction(float(v)) for v in values), Fraction(0))
    f = np.float32(float(s))            # within one float32 ulp of s
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - s), int(c.view(np.uint32)) & 1))
    return best


def pin_router_one_hot_rows(router_logits):
    """W_r[e] = e-th unit vector: logits = round_f32(x[t, e] + b[e])."""
    rng = np.random.default_rng(31)
    T, H, E = 3, 16, 10
    x = to_bits(rng.standard_normal((T, H)))
    w = np.zeros((E, H), np.float32)
    w[np.arange(E), np.arange(E)] = 1.0
    b = rng.standard_normal(E).astype(np.float32)
    got = router_logits(x, to_bits(w), b)
    xf = from_bits(x)
    want = np.float32(xf[:, :E] + b.astype(np.float64)[None, :])  # the sum is exact in float64
    assert np.array_equal(got, want)


def pin_router_small_integers_match_matmul(router_logits):
    """Small-integer inputs: every product and partial sum is an exact
    integer, so a library matmul in float64 is the exact answer."""
    rng = np.random.default_rng(32)
    T, H, E = 5, 48, 7
    x = rng.integers(-4, 5, (T, H)).astype(np.float32)
    w = rng.integers(-4, 5, (E, H)).astype(np.float32)
    b = rng.integers(-8, 9, E).astype(np.float32)
    got = router_logits(to_bits(x), to_bits(w), b)
    want = (x.astype(np.float64) @ w.astype(np.float64).T + b).astype(np.float32)
    assert np.array_equal(got, want)
    assert np.array_equal(router_logits(to_bits(x), to_bits(w), None),
                          (x.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32))


def pin_router_cancellation(router_logits):
    """2^24 + 1 - 2^24 = 1 exactly (a float32 running sum returns 0)."""
    x = to_bits(np.float32([[2.0 ** 24, 1.0, -(2.0 ** 24), 0.0]]))
    w = to_bits(np.ones((2, 4), np.float32))
    got = router_logits(x, w, np.float32([0.0, 0.5]))
    assert got.tolist() == [[1.0, 1.5]]


def pin_router_double_rounding(router_logits):
    """The exact sum 1 + 2^-24 + 2^-80 lies just above the float32 midpoint
    between 1 and 1 + 2^-23, so it rounds up; rounding it to float64 first
    lands on the midpoint, which ties to even (1.0)."""
    x = to_bits(np.float64([[1.0, 2.0 ** -12, 2.0 ** -40]]))
    w = to_bits(np.float64([[1.0, 2.0 ** -12, 2.0 ** -40]]))
    got = router_logits(x, w, None)
    assert got[0, 0] == np.nextafter(np.float32(1.0), np.float32(2.0))
    # and exactly at the midpoint: ties to even
    x2 = to_bits(np.float64([[1.0, 2.0 ** -12]]))
    assert router_logits(x2, x2, None)[0, 0] == np.float32(1.0)


def pin_router_random_against_exact_rationals(router_logits):
    """Random BF16 inputs of mixed magnitudes, rectangular W_r: every logit
    equals the exact rational sum rounded to float32 by hand."""
    rng = np.random.default_rng(33)
    T, H, E = 2, 24, 5
    x = to_bits(rng.standard_normal((T, H)) * np.exp2(rng.integers(-12, 12, (T, H))))
    w = to_bits(rng.standard_normal((E, H)) * np.exp2(rng.integers(-12, 12, (E, H))))
    b = (rng.standard_normal(E) * 3).astype(np.float32)
    got = router_logits(x, w, b)
    xf, wf = from_bits(x), from_bits(w)
    for t in range(T):
        for e in range(E):
            want = _exact_f32([*(xf[t] * wf[e]).tolist(), float(b[e])])
            assert got[t, e] == want, (t, e, got[t, e], want)


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_")]
