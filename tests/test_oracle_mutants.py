"""Plant plausible mistakes in a copy of the oracle source and check that at
least one pin catches each.  The mistakes are planted in the oracle, on the
CPU; the product is not involved."""
import os

import pytest

import oracle
from oracle import build as obuild
from tests import _pins

SRC = open(os.path.join(os.path.dirname(obuild.__file__), "kvc_oracle.c")).read()

MUTANTS = {
    "scale_1_over_d": ("1.0 / sqrt((double)d_h)", "1.0 / (double)d_h"),
    "interleaved_groups": ("const int32_t kv = h / g;", "const int32_t kv = h % H_kv;"),
    "drops_newest_row": ("for (int64_t j = 0; j < n; ++j) {\n                double dot",
                         "for (int64_t j = 0; j < n - 1; ++j) {\n                double dot"),
    "keys_for_values": ("acc[d] += w[j] * load_elem(V,", "acc[d] += w[j] * load_elem(K,"),
    "sign_of_exponent": ("w[j] = exp(w[j] - m);", "w[j] = exp(m - w[j]);"),
    "no_normalisation": ("out[qrow + d] = acc[d] / denom;", "out[qrow + d] = acc[d];"),
    "bf16_shift": ("(uint32_t)h << 16", "(uint32_t)h << 15"),
    "fp16_bias": ("expo - 25", "expo - 24"),
    "reversed_query": ("load_elem(q, qrow + d, dtype)", "load_elem(q, qrow + (d_h - 1 - d), dtype)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found exactly once"
    lib = oracle.load_library(obuild.build_variant(SRC.replace(old, new), name))
    caught = []
    for pin in _pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
