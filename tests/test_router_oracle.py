"""The oracle's router projection against its pins, and planted mistakes in
copies of it that each must trip a pin (CPU only)."""
import importlib.util
import os

import pytest

import oracle
from oracle import router as committed
from tests import router_pins

pytestmark = pytest.mark.cpu

SOURCE = os.path.join(os.path.dirname(oracle.__file__), "router.py")

MUTANTS = {
    "bias_dropped": ("[*prods.tolist(), float(b[e])]", "[*prods.tolist(), 0.0]"),
    "float32_running_sum": ("out[t, e] = round_f32_exact([*prods.tolist(), float(b[e])])",
                            "out[t, e] = np.float32(prods.astype(np.float32).sum(dtype=np.float32) + np.float32(b[e]))"),
    "double_rounding_kept": ("    if Fraction(s) != mid:\n        return f", "    if True:\n        return f"),
    "wrong_weight_row": ("prods = x[t] * w[e]", "prods = x[t] * w[(e + 1) % E]"),
}


@pytest.mark.parametrize("pin", router_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(committed.router_logits)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "router_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("router_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    failed = []
    for pin in router_pins.ALL_PINS:
        try:
            pin(mod.router_logits)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
