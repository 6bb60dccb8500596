"""Pins of the layer prologue/epilogue oracle (oracle/layer.py) against facts
that do not come from the oracle itself: a hand-computed convolution,
causality and left padding, the unit norm of L2-normalised rows, sigmoid and
RMS-norm closed forms, and the decay range the operator expects."""
import numpy as np

from oracle import layer


def test_short_conv_hand_example():
    """One channel, W = 3, taps (a, b, c) = (0.5, -1, 2) on x = (1, 2, 3, 4):
    y_t = 2 x_t - x_{t-1} + 0.5 x_{t-2}, with zeros before the start."""
    x = np.array([1.0, 2.0, 3.0, 4.0]).reshape(4, 1, 1)
    w = np.array([0.5, -1.0, 2.0]).reshape(1, 1, 3)
    y = layer.short_conv(x, w)[:, 0, 0]
    assert np.allclose(y, [2.0, 3.0, 4.5, 6.0], rtol=0, atol=1e-15)


def test_short_conv_is_causal_and_left_padded_per_sequence():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((12, 2, 5))
    w = rng.standard_normal((2, 5, 4))
    cu = [0, 5, 5, 12]  # the middle sequence is empty
    y = layer.short_conv(x, w, cu)
    x2 = x.copy()
    x2[8] += 100.0  # a later token of sequence 2 changes only tokens >= 8 of it
    y2 = layer.short_conv(x2, w, cu)
    assert np.array_equal(y[:8], y2[:8])
    assert not np.allclose(y[8:12], y2[8:12])
    x3 = x.copy()
    x3[4] += 100.0  # the last token of sequence 0 never reaches sequence 2
    assert np.array_equal(layer.short_conv(x3, w, cu)[5:], y[5:])
    # the first token of a sequence sees only itself (the last tap)
    assert np.allclose(y[5], w[:, :, -1] * x[5], rtol=0, atol=1e-15)


def test_short_conv_width_one_is_a_scale():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 3, 4))
    w = rng.standard_normal((3, 4, 1))
    assert np.allclose(layer.short_conv(x, w), x * w[:, :, 0], rtol=0, atol=1e-15)


def test_l2_rows_have_unit_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((9, 3, 128)) * 10
    n = np.linalg.norm(layer.l2_normalise(x), axis=-1)
    assert np.allclose(n, 1.0, rtol=0, atol=1e-9)
    z = layer.l2_normalise(np.zeros((1, 1, 8)))  # the eps keeps zero rows finite
    assert np.all(z == 0.0)


def test_gates_closed_forms_and_range():
    a = np.array([-50.0, -1.0, 0.0, 1.0, 50.0])
    q, k, v, g, beta = layer.prologue(np.ones((5, 1, 2)), np.ones((5, 1, 2)),
                                      np.ones((5, 1, 2)), a[:, None, None] * np.ones((5, 1, 2)),
                                      a[:, None], np.ones((1, 2, 1)), np.ones((1, 2, 1)),
                                      np.ones((1, 2, 1)))
    assert np.allclose(beta[:, 0], [1 / (1 + np.exp(50)), 1 / (1 + np.e), 0.5,
                                    1 / (1 + np.exp(-1)), 1 / (1 + np.exp(-50))])
    assert np.allclose(g[2], -2.5) and np.all(g <= 0) and np.all(g >= -5)


def test_epilogue_closed_forms():
    """A constant row c has RMS |c|: it becomes sign(c) w sigmoid(gate); a zero
    gate halves it."""
    o = np.full((2, 1, 4), -3.0)
    w = np.array([1.0, 2.0, 0.5, -1.0])
    y = layer.epilogue(o, np.zeros((2, 1, 4)), w, eps=0.0)
    assert np.allclose(y[0, 0], -w * 0.5, rtol=0, atol=1e-15)
    rng = np.random.default_rng(3)
    o = rng.standard_normal((5, 2, 16))
    y = layer.epilogue(o, np.full((5, 2, 16), 60.0), np.ones(16))  # gate ~ 1
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-5)
