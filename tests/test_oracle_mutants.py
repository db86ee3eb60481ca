"""Planted mistakes in copies of the oracle must each trip at least one pin.

Each mutant is a text substitution applied to a temporary copy of
oracle/moe_oracle.c, compiled with the same gcc flags.  The committed oracle
is never modified.  A mutant that passes every pin would mean the pins cannot
tell that mistake from the definition.
"""
import os

import pytest

import oracle
from tests import oracle_pins

pytestmark = pytest.mark.cpu

MUTANTS = {
    "tie_to_higher_index": ("logits[e] > logits[best]", "logits[e] >= logits[best]"),
    "silu_sign": ("g / (1.0 + exp(-g))", "g / (1.0 + exp(g))"),
    "gate_up_swapped": ("double silu_g = g / (1.0 + exp(-g));\n        a[i] = silu_g * u;",
                        "double silu_g = u / (1.0 + exp(-u));\n        a[i] = silu_g * g;"),
    "down_transposed": ("acc += bf16_to_double(down_row[i]) * a[i];",
                        "acc += bf16_to_double(wd_e[i * H + h]) * a[i];"),
    "combine_weight_dropped": ("out[h] += w[j] * y[h];", "out[h] += y[h];"),
    "softmax_unnormalised": ("w[j] = w[j] / s;", "w[j] = w[j];"),
    "up_row_off_by_one": ("wgu_e + (I + i) * H", "wgu_e + (I + i - 1) * H"),
    "x_reversed": ("double xh = bf16_to_double(x[h]);", "double xh = bf16_to_double(x[H - 1 - h]);"),
    "last_slot_dropped": ("for (int64_t j = 0; j < k; ++j) {\n            int64_t blk",
                          "for (int64_t j = 0; j + 1 < k; ++j) {\n            int64_t blk"),
    "bf16_low_half": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "softmax_max_not_first": ("double m = (double)logits[idx[0]];", "double m = 0.0 * (double)logits[idx[0]] + 1.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mpath), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    if name == "softmax_max_not_first":
        # shifting by a constant other than the max is mathematically the same
        # softmax; this "mutant" is a control that the pins must NOT reject
        assert failed == [], failed
    else:
        assert failed, f"no pin caught mutant {name}"
