"""The backward oracle against its pins (tests/backward_pins.py), and planted
mistakes in copies of the oracle, each of which must trip at least one pin.
The committed oracle is never modified: each mutant is a text substitution
in a temporary copy of oracle/moe_backward.py, loaded as a module of its own."""
import importlib.util

import numpy as np
import pytest

import oracle
from oracle import moe_backward as bwd_mod
from tests import backward_pins

pytestmark = pytest.mark.cpu


def _bound(f):
    return lambda x, L, wgu, wd, dout, k, **kw: f(x, L, wgu, wd, dout, k, oracle.route, **kw)


@pytest.mark.parametrize("pin", backward_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_backward_pin(pin):
    pin(oracle.backward)


def test_backward_is_the_sum_of_expert_parts():
    # the per-expert step on one expert's rows gives that expert's gradients
    rng = np.random.default_rng(31)
    x, L, wgu, wd = backward_pins.rand_layer(rng, 6, 32, 16, 5)
    dout = backward_pins.rand_dout(rng, 6, 32)
    full = oracle.backward(x, L, wgu, wd, dout, 2)
    xf, df = bwd_mod.bf16_to_f64(x), dout.astype(np.float64)
    for e in np.unique(full["idx"]):
        tok, slot = np.nonzero(full["idx"] == e)
        _, dw, dwgu, dwd = bwd_mod.expert_backward(xf[tok], df[tok], full["w"][tok, slot], wgu[e], wd[e])
        assert np.array_equal(dwgu, full["dwgu"][e]) and np.array_equal(dwd, full["dwd"][e])
        assert np.array_equal(dw, full["dw"][tok, slot])


def test_backward_expert_map_matches_full():
    # only the selected experts' blocks passed: the same gradients for them
    rng = np.random.default_rng(30)
    x, L, wgu, wd = backward_pins.rand_layer(rng, 5, 32, 16, 10)
    dout = backward_pins.rand_dout(rng, 5, 32)
    full = oracle.backward(x, L, wgu, wd, dout, 3)
    used = np.unique(full["idx"])
    emap = -np.ones(10, np.int32)
    emap[used] = np.arange(len(used), dtype=np.int32)
    part = oracle.backward(x, L, wgu[used], wd[used], dout, 3, expert_map=emap)
    for name in ("dx", "dlogits"):
        assert np.array_equal(part[name], full[name])
    assert np.array_equal(part["dwgu"], full["dwgu"][used])
    assert np.array_equal(part["dwd"], full["dwd"][used])


MUTANTS = {
    "silu_derivative_term_dropped": ("dg = da * u * s * (1.0 + g * (1.0 - s))", "dg = da * u * s"),
    "du_without_gate": ("du = da * g * s", "du = da * s"),
    "dx_up_term_dropped": ("dx_rows = dg @ Wg + du @ Wu", "dx_rows = dg @ Wg"),
    "dwd_weight_dropped": ("dwd = (we[:, None] * de).T @ a", "dwd = de.T @ a"),
    "dlogits_sign": ("w * (dw - S[:, None])", "w * (S[:, None] - dw)"),
    "dlogits_centering_dropped": ("w * (dw - S[:, None])", "w * dw"),
    "q_reversed": ("q = de @ Wd ", "q = (de @ Wd)[:, ::-1] "),
    "dwgu_gate_up_swapped": ("np.concatenate([dg.T @ xe, du.T @ xe])", "np.concatenate([du.T @ xe, dg.T @ xe])"),
    "da_weight_dropped": ("da = we[:, None] * q", "da = q"),
    "gate_up_swapped": ("g = xe @ Wg.T\n    u = xe @ Wu.T", "g = xe @ Wu.T\n    u = xe @ Wg.T"),
    "dw_not_reduced_over_neurons": ("dw = np.sum(a * q, axis=1)", "dw = a[:, 0] * q[:, 0]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(bwd_mod.__file__).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant_backward.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"mutant_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    f = _bound(mod.backward)
    failed = []
    for pin in backward_pins.ALL_PINS:
        try:
            pin(f)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
