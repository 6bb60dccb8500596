"""Pins for the fp64 oracle, against what the pages and the mathematics fix.

Each test below would fail for a plausible slip in the oracle: a dropped or
misplaced decay, decay applied after the write, the erase read through S
instead of S^T, the output taken from the state before the update, a missing
clamp or scale, a wrong sign on the erase.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests.chunked_fp64 import chunked_prefill, gram_subtile, _gram_direct

GOLD = os.path.join(os.path.dirname(__file__), "golden")

# The prefill under test. tests/test_oracle_mutations.py swaps in oracle
# builds with planted mistakes and checks that these pins catch each one.
_PF = [oracle.prefill]


def PF(*args, **kw):
    return _PF[0](*args, **kw)


def rnd_inputs(rng, T, H, Dk, Dv, g_lo=-5.0, unit=True):
    q = rng.standard_normal((T, H, Dk))
    k = rng.standard_normal((T, H, Dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, Dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    g = g_lo * (1.0 / (1.0 + np.exp(-rng.standard_normal((T, H, Dk)))))
    f = lambda x: x.astype(np.float32)
    return f(q), f(k), f(v), f(g), f(beta)


def exact_unit_keys(rng, T, H, D, support=4):
    """Keys of exactly unit norm in float32: +-1/sqrt(support) on `support`
    random channels, with support a power of 4 (entries are powers of two)."""
    k = np.zeros((T, H, D), dtype=np.float32)
    val = np.float32(1.0 / math.sqrt(support))
    for t in range(T):
        for h in range(H):
            idx = rng.choice(D, size=support, replace=False)
            k[t, h, idx] = val * rng.choice([-1.0, 1.0], size=support)
    return k


def test_hand_worked_example():
    """Golden values derived by hand (tests/golden/delta_rule_worked_example.json)."""
    with open(os.path.join(GOLD, "delta_rule_worked_example.json")) as f:
        G = json.load(f)
    E = math.exp(-5.0)
    q = np.array(G["q"], dtype=np.float32)[:, None, :]
    k = np.array(G["k"], dtype=np.float32)[:, None, :]
    v = np.array(G["v"], dtype=np.float32)[:, None, :]
    g = np.array(G["g"], dtype=np.float32)[:, None, :]
    beta = np.array(G["beta"], dtype=np.float32)[:, None]
    out, fin = PF(q, k, v, g, beta, G["scale"])
    want_o = np.array(G["out_const"]) + E * np.array(G["out_coefE"])
    want_s = np.array(G["final_const"]) + E * np.array(G["final_coefE"])
    # inputs 0.6, 0.8, ln(1/2), ln(1/4) are float32-rounded: ~1e-7 relative
    np.testing.assert_allclose(out[:, 0, :], want_o, rtol=0, atol=2e-7)
    np.testing.assert_allclose(fin[0, 0], want_s, rtol=0, atol=2e-7)


@pytest.mark.parametrize("Dk,Dv", [(4, 3), (16, 16), (128, 128)])
def test_delta_invariant_unit_key_beta_one(Dk, Dv):
    """||k||=1, beta=1: the write makes S_t^T k_t = v_t exactly, for any decay
    ('Kimi K3...' section DeltaNet: the stale association S^T k - v is
    removed). With q_t = k_t the output is therefore scale * v_t."""
    rng = np.random.default_rng(11)
    T, H = 40, 2
    support = 4 if Dk < 16 else 16
    k = exact_unit_keys(rng, T, H, Dk, support)
    _, _, v, g, _ = rnd_inputs(rng, T, H, Dk, Dv, g_lo=-6.0)
    beta = np.ones((T, H), dtype=np.float32)
    S0 = rng.standard_normal((1, H, Dk, Dv))
    out, fin = PF(k, k, v, g, beta, 0.5, init_state=S0)
    np.testing.assert_allclose(out, 0.5 * v.astype(np.float64), rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.einsum("hij,hi->hj", fin[0], k[-1].astype(np.float64)),
                               v[-1].astype(np.float64), rtol=0, atol=1e-12)


def test_beta_zero_is_pure_decay_with_clamp():
    """beta=0 removes erase and write: S_t = Diag(exp(sum clamp(g))) S0 and
    o_t = scale * S_t^T q_t. g spans [-9, +3] to exercise the clamp to
    [-5, 0] ('K3 vs DSV4...', section 硬件适配)."""
    rng = np.random.default_rng(3)
    T, H, Dk, Dv = 17, 3, 8, 5
    q, k, v, _, _ = rnd_inputs(rng, T, H, Dk, Dv)
    g = rng.uniform(-9.0, 3.0, size=(T, H, Dk)).astype(np.float32)
    beta = np.zeros((T, H), dtype=np.float32)
    S0 = rng.standard_normal((1, H, Dk, Dv))
    out, fin = PF(q, k, v, g, beta, 0.25, init_state=S0)
    gc = np.clip(g.astype(np.float64), -5.0, 0.0)
    cum = np.cumsum(gc, axis=0)
    for t in range(T):
        St = np.exp(cum[t])[:, :, None] * S0[0]
        np.testing.assert_allclose(out[t], 0.25 * np.einsum("hij,hi->hj", St, q[t].astype(np.float64)),
                                   rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fin[0], np.exp(cum[-1])[:, :, None] * S0[0], rtol=1e-12, atol=1e-14)


def test_one_hot_distinct_keys_is_gated_linear_attention():
    """Pairwise-distinct one-hot keys and S0 = 0: every earlier write sits on
    another key channel, so S^T k_t = 0 before the write and KDA reduces to
    gated linear attention with beta-scaled values ('Kimi K3...', sections
    '线性注意力' and 'Gated DeltaNet'): S_t = Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T."""
    rng = np.random.default_rng(5)
    T, H, D = 12, 2, 16
    q, _, v, g, beta = rnd_inputs(rng, T, H, D, D)
    k = np.zeros((T, H, D), dtype=np.float32)
    for h in range(H):
        k[np.arange(T), h, rng.permutation(D)[:T]] = 1.0
    out, fin = PF(q, k, v, g, beta, 0.3)
    for h in range(H):
        S = np.zeros((D, D))
        for t in range(T):
            alpha = np.exp(np.clip(g[t, h].astype(np.float64), -5, 0))
            S = alpha[:, None] * S + float(beta[t, h]) * np.outer(k[t, h].astype(np.float64), v[t, h].astype(np.float64))
            np.testing.assert_allclose(out[t, h], 0.3 * S.T @ q[t, h].astype(np.float64),
                                       rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(fin[0, h], S, rtol=1e-12, atol=1e-14)


def test_scalar_gate_is_gated_deltanet_matrix_form():
    """All channels sharing one log-decay is Gated DeltaNet ('Kimi K3...',
    section 'Gated DeltaNet': a scalar forget gate alpha on S); checked
    against the product form S_t = alpha_t (I - beta k k^T) S + beta k v^T."""
    rng = np.random.default_rng(9)
    T, H, Dk, Dv = 20, 2, 8, 6
    q, k, v, _, beta = rnd_inputs(rng, T, H, Dk, Dv)
    gs = (-3.0 * rng.random((T, H))).astype(np.float32)
    g = np.repeat(gs[:, :, None], Dk, axis=2)
    S0 = rng.standard_normal((1, H, Dk, Dv))
    out, fin = PF(q, k, v, g, beta, 1.0, init_state=S0)
    for h in range(H):
        S = S0[0, h].copy()
        for t in range(T):
            kk = k[t, h].astype(np.float64)
            b = float(beta[t, h])
            S = math.exp(float(gs[t, h])) * (np.eye(Dk) - b * np.outer(kk, kk)) @ S + b * np.outer(kk, v[t, h].astype(np.float64))
            np.testing.assert_allclose(out[t, h], S.T @ q[t, h].astype(np.float64), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], S, rtol=1e-11, atol=1e-12)


def test_key_channel_permutation():
    """Permuting the key channels of q, k, g and the rows of S0 together
    leaves o unchanged and permutes the rows of the final state (any g)."""
    rng = np.random.default_rng(21)
    T, H, Dk, Dv = 30, 2, 12, 7
    q, k, v, g, beta = rnd_inputs(rng, T, H, Dk, Dv)
    S0 = rng.standard_normal((1, H, Dk, Dv))
    p = rng.permutation(Dk)
    o1, f1 = PF(q, k, v, g, beta, 0.7, init_state=S0)
    o2, f2 = PF(q[..., p], k[..., p], v, g[..., p], beta, 0.7, init_state=S0[:, :, p, :])
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(f2, f1[:, :, p, :], rtol=1e-12, atol=1e-13)


def test_erase_is_non_expansive():
    """With ||k|| = 1, beta in [0, 1] and alpha in (0, 1], the map
    S -> (I - beta k k^T) Diag(alpha) S is non-expansive, so two runs that
    differ only in S0 never move apart (an erase with the wrong sign would)."""
    rng = np.random.default_rng(4)
    T, H, D = 50, 1, 16
    q, k, v, g, beta = rnd_inputs(rng, T, H, D, D)
    S0a = rng.standard_normal((1, H, D, D))
    S0b = S0a + rng.standard_normal((1, H, D, D))
    prev = np.linalg.norm(S0a - S0b)
    for t in range(1, T + 1):
        _, fa = PF(q[:t], k[:t], v[:t], g[:t], beta[:t], 1.0, init_state=S0a)
        _, fb = PF(q[:t], k[:t], v[:t], g[:t], beta[:t], 1.0, init_state=S0b)
        cur = np.linalg.norm(fa - fb)
        assert cur <= prev * (1 + 1e-6) + 1e-12
        prev = cur
    assert prev < 0.5 * np.linalg.norm(S0a - S0b)


def test_token_order_matters():
    """The delta recurrence does not commute ('K3 vs DSV4...': the recurrence
    carries position), so reversing two tokens changes the result."""
    rng = np.random.default_rng(8)
    q, k, v, g, beta = rnd_inputs(rng, 6, 1, 8, 8)
    _, f1 = PF(q, k, v, g, beta, 1.0)
    idx = [0, 1, 2, 4, 3, 5]
    _, f2 = PF(q[idx], k[idx], v[idx], g[idx], beta[idx], 1.0)
    assert np.max(np.abs(f1 - f2)) > 1e-3


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("T", [5, 64, 70])
def test_chunked_equals_token_recurrence(C, T):
    """Brute force: the chunked form ('Kimi K3...', section FlashKDA 算法)
    reaches the token recurrence in exact arithmetic; in fp64 to ~1e-12."""
    rng = np.random.default_rng(100 + C + T)
    H, Dk, Dv = 2, 8, 6
    q, k, v, g, beta = rnd_inputs(rng, T, H, Dk, Dv)
    S0 = rng.standard_normal((1, H, Dk, Dv))
    out, fin = PF(q, k, v, g, beta, 0.5, init_state=S0)
    for h in range(H):
        o, S = chunked_prefill(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], 0.5, S0[0, h], C)
        np.testing.assert_allclose(o, out[:, h], rtol=0, atol=1e-11)
        np.testing.assert_allclose(S, fin[0, h], rtol=0, atol=1e-11)


@pytest.mark.parametrize("g_lo", [-5.0, -50.0])
def test_subtile_factorisation_matches_direct_decay(g_lo):
    """The bf16-safe factorisation of the chunk Gram matrices through
    16-token tile references equals the element-wise decay form, including
    at the decay floor (g = -5 everywhere after clamping)."""
    rng = np.random.default_rng(77)
    C, D = 64, 16
    x = rng.standard_normal((C, D))
    k = rng.standard_normal((C, D))
    g = np.clip(g_lo * rng.random((C, D)), -5, 0)
    a = np.cumsum(g, axis=0)
    for strict in (False, True):
        ref = _gram_direct(x, k, a, strict)
        got = gram_subtile(x, k, a, strict=strict)
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-300)
    # the row factors are <= 1 and the column factors stay below e^80
    r = a[15]
    assert np.all(np.exp(r - a[16:32]) <= np.exp(80.0) * (1 + 1e-12))


def test_chunked_subtile_equals_token_recurrence_at_floor():
    rng = np.random.default_rng(31)
    T, Dk, Dv = 130, 8, 8
    q, k, v, _, beta = rnd_inputs(rng, T, 1, Dk, Dv)
    g = np.full((T, 1, Dk), -5.0, dtype=np.float32)
    S0 = rng.standard_normal((1, 1, Dk, Dv))
    out, fin = PF(q, k, v, g, beta, 1.0, init_state=S0)
    o, S = chunked_prefill(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], 1.0, S0[0, 0], 64, subtile=True)
    np.testing.assert_allclose(o, out[:, 0], rtol=0, atol=1e-10)
    np.testing.assert_allclose(S, fin[0, 0], rtol=0, atol=1e-10)


def test_split_resume_and_varlen_packing():
    """prefill(T1 + T2) == prefill(T2, init = final(T1)); packed sequences
    equal separate calls; a zero-length sequence leaves its state as given."""
    rng = np.random.default_rng(12)
    H, D = 2, 8
    q, k, v, g, beta = rnd_inputs(rng, 45, H, D, D)
    S0 = rng.standard_normal((1, H, D, D))
    o_all, f_all = PF(q, k, v, g, beta, 0.5, init_state=S0)
    o1, f1 = PF(q[:19], k[:19], v[:19], g[:19], beta[:19], 0.5, init_state=S0)
    o2, f2 = PF(q[19:], k[19:], v[19:], g[19:], beta[19:], 0.5, init_state=f1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o_all, rtol=0, atol=1e-12)
    np.testing.assert_allclose(f2, f_all, rtol=0, atol=1e-12)

    cu = [0, 19, 19, 45]
    init3 = np.concatenate([S0, 2 * S0, S0], axis=0)
    o3, f3 = PF(q, k, v, g, beta, 0.5, init_state=init3, cu_seqlens=cu)
    oB, fB = PF(q[19:], k[19:], v[19:], g[19:], beta[19:], 0.5, init_state=S0)
    np.testing.assert_allclose(o3[:19], o1, rtol=0, atol=0)
    np.testing.assert_allclose(o3[19:], oB, rtol=0, atol=0)
    np.testing.assert_array_equal(f3[1], 2 * S0[0])
    np.testing.assert_allclose(f3[2], fB[0], rtol=0, atol=0)


def test_decode_steps_equal_prefill():
    """T single-token decode steps reproduce one T-token prefill
    ('Kimi K3...', section FlashKDA 算法: decode follows the recurrence)."""
    rng = np.random.default_rng(13)
    B, H, D, T = 3, 2, 8, 9
    q, k, v, g, beta = rnd_inputs(rng, T * B, H, D, D)
    S = rng.standard_normal((B, H, D, D))
    sh = lambda x: x.reshape(B, T, *x.shape[1:])
    qs, ks, vs, gs, bs = map(sh, (q, k, v, g, beta))
    outs = []
    state = S.copy()
    for t in range(T):
        o, state = PF(qs[:, t], ks[:, t], vs[:, t], gs[:, t], bs[:, t], 0.5, init_state=state,
                      cu_seqlens=np.arange(B + 1))
        outs.append(o)
    flat = lambda x: x.reshape(B * T, *x.shape[2:])
    op, fp = PF(flat(qs), flat(ks), flat(vs), flat(gs), flat(bs), 0.5, init_state=S,
                            cu_seqlens=np.arange(B + 1) * T)
    np.testing.assert_allclose(np.stack(outs, 1).reshape(B * T, H, D), op, rtol=0, atol=1e-12)
    np.testing.assert_allclose(state, fp, rtol=0, atol=1e-12)


def test_oracle_rejects_bad_cu_seqlens():
    rng = np.random.default_rng(1)
    q, k, v, g, beta = rnd_inputs(rng, 8, 1, 4, 4)
    with pytest.raises(ValueError):
        PF(q, k, v, g, beta, 1.0, cu_seqlens=np.array([0, 5, 3, 8]))


def test_decode_step_wrapper():
    rng = np.random.default_rng(14)
    q, k, v, g, beta = rnd_inputs(rng, 4, 2, 8, 8)
    S = rng.standard_normal((4, 2, 8, 8))
    o1, s1 = oracle.decode_step(q, k, v, g, beta, 0.5, S)
    o2, s2 = oracle.prefill(q, k, v, g, beta, 0.5, init_state=S, cu_seqlens=np.arange(5))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)
