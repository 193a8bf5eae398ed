"""Plant plausible mistakes in a copy of the oracle (CPU only) and check that the pins catch each.

This guards the pins themselves: a dropped term, a wrong sign, operand or index in
the oracle must fail at least one of them.
"""
import os
import subprocess

import pytest

import test_oracle_pins as pins
from oracle import recurrence as orc

SRC = os.path.join(os.path.dirname(orc.__file__), "gdn_oracle.c")

MUTANTS = {
    "no_decay": ("S[e] *= alpha;", "S[e] *= 1.0;"),
    "half_decay": ("const double alpha = exp(gt);", "const double alpha = exp(0.5 * gt);"),
    "delta_sign": ("p[j] = bt * (vt[j] - p[j]);", "p[j] = bt * (vt[j] + p[j]);"),
    "no_beta": ("p[j] = bt * (vt[j] - p[j]);", "p[j] = (vt[j] - p[j]);"),
    "lookup_with_q": ("p[j] += S[(size_t)i * dv + j] * kt[i];", "p[j] += S[(size_t)i * dv + j] * qt[i];"),
    "write_with_q": ("S[(size_t)i * dv + j] += kt[i] * p[j];", "S[(size_t)i * dv + j] += qt[i] * p[j];"),
    "gqa_modulo": ("const int hk = h / group;", "const int hk = h % Hqk;"),
    "no_scale": ("for (int j = 0; j < dv; ++j) ot[j] *= scale;", ""),
    "plain_add_no_beta": ("+= bt * kt[i] * vt[j];", "+= kt[i] * vt[j];"),
}

PINS = [
    pins.test_toy_table_and_reads,
    lambda: [pins.test_toy_overwrite(*a) for a in (("linear", 1, 1.0), ("delta", 0, 1.0), ("gated05", 0, 0.5))],
    lambda: [pins.test_decay_powers(a) for a in ("0.9", "0.5")],
    pins.test_repeated_write_distances,
    lambda: [pins.test_write_invariant(a) for a in (0.7,)],
    pins.test_divergence_with_long_key,
    lambda: pins.test_linear_attention_bruteforce(True),
    pins.test_transposed_update_table,
    pins.test_grouped_heads_follow_repeat_interleave,
    lambda: pins.test_chunk_form_equals_token_loop(16),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", lib_path,
                           str(mutated), "-lm"])
    orc.use_library(orc.bind(lib_path))
    failed = 0
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed += 1
    finally:
        orc.reset_library()
    assert failed > 0, f"no pin caught the planted mistake {name!r}"
