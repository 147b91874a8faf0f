"""Pins for the oracle's input pre-processing (oracle.preprocess).

Source: "22580: от GPT-2 до Kimi K3" (temp07.ru), section "DeltaNet, или Fast
Weight Programmers", the forward with a per-token write strength: q and k pass
through SiLU and then F.normalize over the key dimension; beta is the sigmoid of
a projected logit.  Each pin checks a fact fixed by those definitions, not the
formula retyped: closed-form values of SiLU and the sigmoid, the reflection
identities silu(x) - silu(-x) = x and sigmoid(x) + sigmoid(-x) = 1, unit norm and
direction of the normalised rows, F.normalize's zero-row rule, scale invariance,
the order silu -> norm, and the read-back identity of the recurrence ("Kimi Delta
Attention (KDA)", DeltaNet section: with alpha = beta = 1 and a unit key the state
returns v exactly) reached through the normalisation of arbitrary keys.
"""
import math

import numpy as np

import oracle


def test_silu_and_sigmoid_closed_forms():
    ln3 = math.log(3.0)
    x = np.array([[0.0, ln3, -ln3, 60.0, -60.0, 1000.0, -1000.0]])
    q, k, b = oracle.preprocess(x, x, x[0], qk_silu=True, beta_sigmoid=True)
    # sigmoid(ln 3) = 3 / 4, sigmoid(-ln 3) = 1 / 4
    np.testing.assert_allclose(q[0, :3], [0.0, 0.75 * ln3, -0.25 * ln3], rtol=1e-15, atol=0)
    np.testing.assert_allclose(b[:3], [0.5, 0.75, 0.25], rtol=1e-15, atol=0)
    np.testing.assert_array_equal(q, k)
    # saturation without overflow: silu(x) -> x, silu(-x) -> 0, sigmoid -> 1 and 0
    assert np.all(np.isfinite(q)) and np.all(np.isfinite(b))
    np.testing.assert_allclose(q[0, [3, 5]], [60.0, 1000.0], rtol=1e-15)
    assert abs(q[0, 4]) < 1e-24 and q[0, 6] == 0.0
    assert b[5] == 1.0 and b[6] == 0.0


def test_reflection_identities():
    rng = np.random.default_rng(20)
    x = rng.standard_normal((50, 3, 16)) * 4
    sp, _, bp = oracle.preprocess(x, x, x, qk_silu=True, beta_sigmoid=True)
    sm, _, bm = oracle.preprocess(-x, -x, -x, qk_silu=True, beta_sigmoid=True)
    np.testing.assert_allclose(sp - sm, x, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(bp + bm, np.ones_like(x), rtol=1e-15, atol=1e-15)


def test_normalised_rows_are_unit_and_keep_direction():
    rng = np.random.default_rng(21)
    q = rng.standard_normal((40, 2, 32)) * rng.uniform(0.01, 100, (40, 2, 1))
    k = rng.standard_normal((40, 2, 32)) * 7
    qn, kn, _ = oracle.preprocess(q, k, np.zeros((40, 2)), qk_l2norm=True)
    np.testing.assert_allclose(np.linalg.norm(qn, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(kn, axis=-1), 1.0, rtol=1e-14)
    # same direction: the cosine with the raw row is 1
    cos = np.sum(qn * q, axis=-1) / np.linalg.norm(q, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-14)
    # positive rescaling of the raw rows changes nothing
    qs, ks, _ = oracle.preprocess(q * 3.5, k * 1e-3, np.zeros((40, 2)), qk_l2norm=True)
    np.testing.assert_allclose(qs, qn, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(ks, kn, rtol=1e-14, atol=1e-15)


def test_zero_row_stays_zero():
    q = np.zeros((2, 1, 8))
    q[1, 0, 3] = 1e-300
    qn, _, _ = oracle.preprocess(q, q, np.zeros((2, 1)), qk_silu=True, qk_l2norm=True)
    assert np.all(qn[0] == 0.0)  # 0 / max(0, eps) = 0, no NaN
    assert np.all(np.isfinite(qn))


def test_silu_comes_before_the_norm():
    # with both steps the result has unit norm; the other order would not
    rng = np.random.default_rng(22)
    x = rng.standard_normal((30, 2, 16)) * 3
    q, k, _ = oracle.preprocess(x, x, np.zeros((30, 2)), qk_silu=True, qk_l2norm=True)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), 1.0, rtol=1e-14)
    wrong = x / np.linalg.norm(x, axis=-1, keepdims=True)
    wrong = wrong / (1 + np.exp(-wrong))
    assert np.max(np.abs(np.linalg.norm(wrong, axis=-1) - 1.0)) > 0.1


def test_normalised_keys_read_back_the_value():
    # alpha = 1, beta = 1 (logit 60 through the sigmoid): S_t^T k^_t = v_t for the
    # normalised key k^_t, whatever the raw key's length
    rng = np.random.default_rng(23)
    T, H, dk, dv = 12, 2, 8, 5
    kraw = rng.standard_normal((T, H, dk)) * rng.uniform(0.1, 30, (T, H, 1))
    q = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    blog = np.full((T, H), 60.0)
    qn, kn, b = oracle.preprocess(q, kraw, blog, qk_l2norm=True, beta_sigmoid=True)
    assert np.all(b == 1.0)
    g = np.zeros((T, H, dk))
    for t in range(1, T + 1):
        _, fin = oracle.kda_fwd(qn[:t], kn[:t], v[:t], g[:t], b[:t], np.array([0, t]))
        for h in range(H):
            np.testing.assert_allclose(fin[0, h].T @ kn[t - 1, h], v[t - 1, h], rtol=1e-12, atol=1e-12)


def test_very_negative_write_logit_only_decays():
    # sigmoid(-800) underflows to 0: nothing is written, the state only decays
    rng = np.random.default_rng(24)
    T, H, d = 10, 2, 6
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    g = -rng.uniform(0, 0.3, (T, H, d))
    S0 = rng.standard_normal((1, H, d, d))
    _, _, b = oracle.preprocess(q, k, np.full((T, H), -800.0), beta_sigmoid=True)
    assert np.all(b == 0.0)
    _, fin = oracle.kda_fwd(q, k, v, g, b, np.array([0, T]), init_state=S0)
    decay = np.exp(np.sum(g, axis=0))  # [H, d]
    np.testing.assert_allclose(fin[0], decay[:, :, None] * S0[0], rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- the gate step
# log alpha = -c softplus(x): the decay alpha in [0, 1] per key channel of "Kimi Delta
# Attention (KDA)" (alpha = 1 keeps, alpha = 0 clears) as the workloads draw it.
def test_gate_closed_forms():
    ln2 = math.log(2.0)
    x = np.array([0.0, math.log(3.0), -math.log(3.0), 40.0, -40.0, 800.0, -800.0])
    g = oracle.gate_from_logits(x)
    # softplus(0) = ln 2; softplus(ln 3) = ln 4; softplus(-ln 3) = ln(4 / 3)
    np.testing.assert_allclose(g[:3], [-ln2, -2 * ln2, -math.log(4.0 / 3.0)], rtol=1e-15)
    # no overflow or loss at the ends: softplus(x) -> x, softplus(-x) -> e^-x
    assert np.all(np.isfinite(g))
    np.testing.assert_allclose(g[[3, 5]], [-40.0, -800.0], rtol=1e-15)
    np.testing.assert_allclose(g[4], -math.exp(-40.0), rtol=1e-14)
    assert g[6] == 0.0 or abs(g[6]) < 1e-300


def test_gate_identities_and_range():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((200, 3, 16)) * 6
    c = 0.37
    gp, gm = oracle.gate_from_logits(x, c), oracle.gate_from_logits(-x, c)
    # softplus(x) - softplus(-x) = x
    np.testing.assert_allclose(gp - gm, -c * x, rtol=1e-13, atol=1e-13)
    # alpha = e^g in (0, 1], decreasing in x, and linear in the scale c
    assert np.all(gp <= 0.0) and np.all(np.exp(gp) > 0.0)
    xs = np.sort(x.ravel())
    assert np.all(np.diff(oracle.gate_from_logits(xs, c)) <= 0.0)
    np.testing.assert_allclose(oracle.gate_from_logits(x, 2 * c), 2 * gp, rtol=1e-15)
    # the recipe of the workloads: -0.1 softplus of a draw equals the stored log decay
    import torch
    t = torch.from_numpy(x[:, 0]).float()
    np.testing.assert_allclose(oracle.gate_from_logits(t, 0.1),
                               (-torch.nn.functional.softplus(t) * 0.1).double().numpy(),
                               rtol=2e-6, atol=1e-7)
