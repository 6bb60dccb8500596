"""Planted mistakes in the layer prologue/epilogue oracle, on the CPU: each
mutant of oracle/layer.py (a plausible slip in a step) must fail at least one
of the pins in test_oracle_layer_pins.py. The oracle itself is never
modified; each mutant is a copy of its source, loaded as a separate module."""
import os
import types

import pytest

import oracle
from tests import test_oracle_layer_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "layer.py")

MUTANTS = {
    # the convolution
    "taps_reversed": ("acc += w[:, :, W - 1 - i] * x[s]", "acc += w[:, :, i] * x[s]"),
    "not_reset_per_sequence": ("if s < t0:", "if s < 0:"),
    "sees_the_next_token": ("s = t - i", "s = t - i + 1 if t - i + 1 < t1 else t - i"),
    # the L2 norm
    "l2_eps_outside_sqrt": ("x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)",
                            "x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)"),
    "l2_over_heads": ("np.sum(x * x, axis=-1, keepdims=True)", "np.sum(x * x, axis=-2, keepdims=True)"),
    # the gates
    "sigmoid_sign": ("1.0 / (1.0 + np.exp(-x))", "1.0 / (1.0 + np.exp(x))"),
    "decay_sign": ("g = -5.0 * sigmoid(alpha_raw)", "g = 5.0 * sigmoid(alpha_raw)"),
    "beta_not_squashed": ("    beta = sigmoid(beta_raw)\n", "    beta = np.asarray(beta_raw, dtype=np.float64)\n"),
    # the output normalisation
    "rms_is_a_sum": ("np.mean(o * o, axis=-1, keepdims=True)", "np.sum(o * o, axis=-1, keepdims=True)"),
    "gate_not_squashed": ("np.asarray(w, dtype=np.float64) * sigmoid(gate_raw)",
                          "np.asarray(w, dtype=np.float64) * np.asarray(gate_raw, dtype=np.float64)"),
    "norm_weight_dropped": ("/ rms * np.asarray(w, dtype=np.float64)", "/ rms"),
}

PINS = [
    pins.test_short_conv_hand_example,
    pins.test_short_conv_is_causal_and_left_padded_per_sequence,
    pins.test_short_conv_width_one_is_a_scale,
    pins.test_l2_rows_have_unit_norm,
    pins.test_gates_closed_forms_and_range,
    pins.test_epilogue_closed_forms,
]


def _load(src, name):
    mod = types.ModuleType("layer_" + name)
    exec(compile(src, "layer_" + name + ".py", "exec"), mod.__dict__)
    return mod


def _failing_pins(mod, monkeypatch):
    monkeypatch.setattr(pins, "layer", mod)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_layer_pins_catch_mutant(monkeypatch, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, (name, old)
    failed = _failing_pins(_load(src.replace(old, new), name), monkeypatch)
    assert failed, "mutant %s passed every layer pin" % name


def test_unmutated_layer_source_passes_the_same_pins(monkeypatch):
    assert not _failing_pins(_load(open(SRC).read(), "same"), monkeypatch)
