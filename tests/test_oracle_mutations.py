"""Planted mistakes in the oracle, on the CPU: each mutant of kda_oracle.c
(a plausible slip in the recurrence) must fail at least one of the pins in
test_oracle_pins.py. The oracle itself is never modified; mutants are
compiled into a temporary directory."""
import functools
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTANTS = {
    "no_clamp_at_floor": ("if (gi < -5.0) gi = -5.0;", ""),
    "no_clamp_at_zero": ("if (gi > 0.0) gi = 0.0;", ""),
    "exp_base_2": ("alpha[i] = exp(gi);", "alpha[i] = exp2(gi);"),
    "erase_reads_S_not_ST": ("acc += S[(size_t)i * Dv + j] * (double)kt[i];",
                             "acc += S[(size_t)j * Dv + i] * (double)kt[i];"),
    "erase_sign": ("u[j] = bt * ((double)vt[j] - acc);", "u[j] = bt * ((double)vt[j] + acc);"),
    "beta_dropped": ("u[j] = bt * ((double)vt[j] - acc);", "u[j] = ((double)vt[j] - acc);"),
    "decay_after_write": (
        "S[(size_t)i * Dv + j] *= alpha[i];",
        "(void)0;",
        "S[(size_t)i * Dv + j] += (double)kt[i] * u[j];",
        "S[(size_t)i * Dv + j] = (S[(size_t)i * Dv + j] + (double)kt[i] * u[j]) * alpha[i];"),
    "output_before_write": ("acc += S[(size_t)i * Dv + j] * (double)qt[i];",
                            "acc += (S[(size_t)i * Dv + j] - (double)kt[i] * u[j]) * (double)qt[i];"),
    "scale_dropped": ("ot[j] = J->scale * acc;", "ot[j] = acc;"),
    "init_state_ignored": ("if (J->init) memcpy", "if (0) memcpy"),
}

PIN_CALLS = [
    pins.test_hand_worked_example,
    functools.partial(pins.test_delta_invariant_unit_key_beta_one, 16, 16),
    pins.test_beta_zero_is_pure_decay_with_clamp,
    pins.test_one_hot_distinct_keys_is_gated_linear_attention,
    pins.test_scalar_gate_is_gated_deltanet_matrix_form,
    functools.partial(pins.test_chunked_equals_token_recurrence, 16, 70),
]


def _build_mutant(tmp_path, name):
    src = open(SRC).read()
    edits = MUTANTS[name]
    for a, b in zip(edits[0::2], edits[1::2]):
        assert src.count(a) >= 1, (name, a)
        src = src.replace(a, b)
    c = tmp_path / (name + ".c")
    c.write_text(src)
    so = tmp_path / (name + ".so")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(c),
                           "-o", str(so), "-lm"])
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    so = _build_mutant(tmp_path, name)
    pins._PF[0] = functools.partial(oracle.prefill, _lib_path=so)
    failed = []
    try:
        for call in PIN_CALLS:
            try:
                call()
            except AssertionError:
                failed.append(getattr(call, "__name__", getattr(call, "func", call).__name__))
    finally:
        pins._PF[0] = oracle.prefill
    assert failed, "mutant %s passed every pin" % name


def test_unmutated_source_passes_the_same_pins(tmp_path):
    src = tmp_path / "same.c"
    src.write_text(open(SRC).read())
    so = tmp_path / "same.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(src),
                           "-o", str(so), "-lm"])
    pins._PF[0] = functools.partial(oracle.prefill, _lib_path=str(so))
    try:
        for call in PIN_CALLS:
            call()
    finally:
        pins._PF[0] = oracle.prefill
