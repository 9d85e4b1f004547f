"""Pins for the oracle of the state-update variants (decay gating, delta rule):
page values, closed forms and brute force. CPU only."""

import json
import os

import numpy as np
import pytest

import oracle as orc
from causal_linear_attention_la_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(B=2, H=3, T=17, dk=4, dv=3, seed=21):
    q, k, v = synth.qkv(B, H, T, dk, dv, seed, dtype="f32")
    return [np.asarray(a, np.float64) for a in (q, k, v)]


# ---------------------------------------------------------------------------
# Decay gating
# ---------------------------------------------------------------------------


def decayed_masked(q, k, v, alpha, eps):
    """Brute force from the definition: o_t = sum_{j<=t} a^(t-j) w_j v_j /
    (sum_{j<=t} a^(t-j) w_j + eps), w_j = phi(q_t).phi(k_j)."""
    phi = orc.FEATURE_MAPS["elu1"][0]
    B, H, T, _ = q.shape
    out = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            a = np.asarray(alpha)[h] if np.ndim(alpha) else alpha
            for t in range(T):
                w = phi(k[b, h, : t + 1]) @ phi(q[b, h, t]) * a ** np.arange(t, -1, -1)
                out[b, h, t] = (w @ v[b, h, : t + 1]) / (w.sum() + eps)
    return out


def test_decay_one_is_the_main_recurrence():
    q, k, v = _rand()
    S0, z0 = np.zeros((2, 3, 4, 3)), np.zeros((2, 3, 4))
    S1, z1, o1 = orc.decode_steps_decay(S0, z0, q, k, v, alpha=1.0)
    S2, z2, o2 = orc.decode_steps(S0, z0, q, k, v)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
    np.testing.assert_array_equal(z1, z2)


@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_decay_matches_weighted_masked_form(eps):
    q, k, v = _rand()
    alpha = np.array([0.5, 0.9, 0.99])          # one factor per head
    _, _, o = orc.decode_steps_decay(np.zeros((2, 3, 4, 3)), np.zeros((2, 3, 4)),
                                     q, k, v, alpha=alpha[None, :], eps=eps)
    np.testing.assert_allclose(o, decayed_masked(q, k, v, alpha, eps), rtol=1e-12, atol=1e-14)


def test_decay_impulse_response():
    """[SSM-LA] section 3: an impulse decays as a^t, for S and for z."""
    for a in (0.5, 0.8, 0.95):
        T = 30
        k = np.zeros((T, 1)); k[0, 0] = 1.0
        v = np.zeros((T, 1)); v[0, 0] = 1.0
        q = np.ones((T, 1))
        S, z = np.zeros((1, 1)), np.zeros(1)
        seq_S = []
        for t in range(T):
            S, z, _ = orc.decode_steps_decay(S, z, q[t:t + 1], k[t:t + 1], v[t:t + 1],
                                             alpha=a, feature="identity")
            seq_S.append(S[0, 0])
            assert z[0] == pytest.approx(a ** t, rel=1e-14)
        np.testing.assert_allclose(seq_S, a ** np.arange(T), rtol=1e-14)
        np.testing.assert_allclose(orc.impulse_response(a, T), a ** np.arange(T), rtol=1e-14)


def test_half_life_table():
    """[SSM-LA] section 3, table '직접 재 보기 C'."""
    g = _load("ssm_decay_half_life.json")
    for a, hl, mem in zip(g["a"], g["half_life_steps"], g["effective_memory"]):
        assert orc.half_life(a) == hl
        total = orc.impulse_response(a, 20000).sum()      # sum of a^t -> 1/(1-a)
        assert round(total) == mem
        assert total == pytest.approx(1.0 / (1.0 - a), rel=1e-9)


# ---------------------------------------------------------------------------
# Delta rule
# ---------------------------------------------------------------------------


def test_delta_rule_page_example():
    """[LA-order]: (5, 3) written under orthogonal keys, then key (0.6, 0.8)
    with value 10: (7.76, 6.68); reads 10 with the key, 7.76 with (1, 0)."""
    g = _load("la_order_delta_rule.json")
    k = np.array(g["k"] + [g["write"]["k"]], float)
    v = np.array(g["v"] + [g["write"]["v"]], float)
    S, out = orc.decode_steps_delta(np.zeros((2, 1)), k[:2], k[:2], v[:2])
    np.testing.assert_array_equal(S[:, 0], g["S_before"])
    S_before = S.copy()
    S, out = orc.decode_steps_delta(S, np.array(g["reads_after"]["queries"][:1], float),
                                    k[2:], v[2:])
    np.testing.assert_allclose(S[:, 0], g["S_after"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(S - S_before, g["difference"] * k[2][:, None], atol=1e-13)
    assert out[0, 0] == pytest.approx(g["reads_after"]["values"][0], abs=1e-13)
    _, o2 = orc.decode_steps_delta(S, np.array([[1.0, 0.0]]), np.zeros((1, 2)), np.zeros((1, 1)))
    assert o2[0, 0] == pytest.approx(g["reads_after"]["values"][1], abs=1e-13)


def test_delta_rule_overwrites_and_orthogonal_writes_add():
    """With unit keys the delta rule overwrites: the read under the key is the
    last value written; a key orthogonal to everything stored adds like the
    plain rule."""
    rng = np.random.default_rng(5)
    kk = rng.standard_normal(6); kk /= np.linalg.norm(kk)
    S = rng.standard_normal((6, 4))
    for val in (rng.standard_normal(4), rng.standard_normal(4)):
        S, out = orc.decode_steps_delta(S, kk[None], kk[None], val[None])
        np.testing.assert_allclose(out[0], val, rtol=1e-12, atol=1e-12)
    e = np.zeros(6); e[0] = 1.0
    S0 = np.zeros((6, 4)); S0[1:] = rng.standard_normal((5, 4))   # nothing under e
    val = rng.standard_normal(4)
    S1, _ = orc.decode_steps_delta(S0, e[None], e[None], val[None])
    np.testing.assert_allclose(S1, S0 + np.outer(e, val), atol=1e-14)


def test_variant_pins_catch_planted_mistakes():
    """Plausible mistakes in the variant oracles fail the pins above."""

    def decayed(S, z, q, k, v, alpha, eps=1e-6, after_add=False, decay_z=True, feature="elu1"):
        f = orc.FEATURE_MAPS[feature][0]
        a = np.asarray(alpha, float)
        out = np.zeros(q.shape[:-1] + (v.shape[-1],))
        for t in range(q.shape[-2]):
            fk, fq = f(k[..., t, :]), f(q[..., t, :])
            if after_add:
                S = a[..., None, None] * (S + fk[..., :, None] * v[..., t, None, :])
                z = a[..., None] * (z + fk)
            else:
                S = a[..., None, None] * S + fk[..., :, None] * v[..., t, None, :]
                z = (a[..., None] if decay_z else 1.0) * z + fk
            out[..., t, :] = np.einsum("...c,...cm->...m", fq, S) / (
                np.einsum("...c,...c->...", fq, z) + eps)[..., None]
        return S, z, out

    # decaying after the add: the impulse pin fails (S_0 = a, not 1)
    T, a = 5, 0.8
    k = np.zeros((T, 1)); k[0, 0] = 1.0
    S, _, _ = decayed(np.zeros((1, 1)), np.zeros(1), np.ones((1, 1)), k[:1], k[:1], a,
                      after_add=True, feature="identity")
    assert S[0, 0] != pytest.approx(1.0)
    # decaying S but not z: the weighted masked form fails
    q, k, v = _rand()
    alpha = np.array([0.5, 0.9, 0.99])
    _, _, o = decayed(np.zeros((2, 3, 4, 3)), np.zeros((2, 3, 4)), q, k, v, alpha[None, :],
                      decay_z=False)
    assert not np.allclose(o, decayed_masked(q, k, v, alpha, 1e-6), rtol=1e-6)

    # a delta rule that forgets to read before writing is the plain rule
    g = _load("la_order_delta_rule.json")
    kk = np.array(g["k"] + [g["write"]["k"]], float)
    vv = np.array(g["v"] + [g["write"]["v"]], float)
    S = np.zeros((2, 1))
    for t in range(3):
        S = S + kk[t][:, None] * vv[t][None, :]
    assert not np.allclose(S[:, 0], g["S_after"], atol=1e-6)


# ---------------------------------------------------------------------------
# Decay-gated backward: alpha = 1 and finite differences of the decayed forward
# ---------------------------------------------------------------------------


def _decay_loss(q, k, v, g, alpha, eps):
    B, H, _, dk = q.shape
    dv = v.shape[-1]
    out = orc.decode_steps_decay(np.zeros((B, H, dk, dv)), np.zeros((B, H, dk)), q, k, v,
                                 alpha=alpha, eps=eps)[2]
    return float(np.sum(g * out))


def _fd_decay(q, k, v, g, alpha, eps, h=1e-6):
    """Central differences of L = sum(g * out) through the decayed forward."""
    grads = []
    for x in (q, k, v):
        gx = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _decay_loss(q, k, v, g, alpha, eps)
            x[idx] = old - h
            lm = _decay_loss(q, k, v, g, alpha, eps)
            x[idx] = old
            gx[idx] = (lp - lm) / (2 * h)
        grads.append(gx)
    return grads


def test_backward_decay_alpha_one_is_plain_backward():
    q, k, v = _rand(T=23, seed=5)
    g = np.random.default_rng(6).standard_normal(v.shape)
    plain = orc.backward_recurrent(q, k, v, g, causal=True)
    decayed = orc.backward_decay(q, k, v, g, alpha=1.0)
    for a, b in zip(decayed, plain):
        assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))


@pytest.mark.parametrize("alpha", [0.5, 0.9, [0.6, 0.97]])
def test_backward_decay_finite_differences(alpha):
    rng = np.random.default_rng(23)
    B, H, N, dk, dv = 1, 2, 6, 3, 4
    q = rng.standard_normal((B, H, N, dk))
    k = rng.standard_normal((B, H, N, dk))
    v = rng.standard_normal((B, H, N, dv))
    g = rng.standard_normal((B, H, N, dv))
    al = np.asarray(alpha, dtype=np.float64)
    al_b = al[None, :] if al.ndim else al      # one factor per head
    eps = 0.05
    fd = _fd_decay(q, k, v, g, al_b, eps)
    got = orc.backward_decay(q, k, v, g, alpha=al_b, eps=eps)
    for a, b in zip(got, fd):
        err = np.max(np.abs(a - b)) / np.max(np.abs(b))
        assert err < 1e-6, err


def test_backward_decay_pins_catch_planted_mistakes():
    """Two plausible mistakes in the reverse sweep, each planted in a copy of
    the oracle's arithmetic, fail the finite-difference pin: the suffix sum
    decayed after adding the token's term (R_j = alpha (phi(q_j) a_j^T +
    R_{j+1})), and no decay on the suffix sums at all."""
    rng = np.random.default_rng(29)
    B, H, N, dk, dv = 1, 1, 5, 2, 3
    q = rng.standard_normal((B, H, N, dk))
    k = rng.standard_normal((B, H, N, dk))
    v = rng.standard_normal((B, H, N, dv))
    g = rng.standard_normal((B, H, N, dv))
    alpha, eps = 0.7, 0.05
    fd = _fd_decay(q, k, v, g, alpha, eps)
    phi, dphi = orc.FEATURE_MAPS["elu1"]
    fq, fk = phi(q[0, 0]), phi(k[0, 0])
    S = np.zeros((dk, dv)); z = np.zeros(dk)
    at = np.zeros((N, dv)); bt = np.zeros(N)
    for t in range(N):
        S = alpha * S + np.outer(fk[t], v[0, 0, t]); z = alpha * z + fk[t]
        D = fq[t] @ z + eps
        o = fq[t] @ S / D
        at[t] = g[0, 0, t] / D; bt[t] = -(g[0, 0, t] @ o) / D

    def dk_with(decay_after_add, decay):
        R = np.zeros((dk, dv)); r = np.zeros(dk); out = np.zeros((N, dk))
        for j in range(N - 1, -1, -1):
            if decay_after_add:
                R = alpha * (R + np.outer(fq[j], at[j])); r = alpha * (r + bt[j] * fq[j])
            else:
                R = decay * R + np.outer(fq[j], at[j]); r = decay * r + bt[j] * fq[j]
            out[j] = (R @ v[0, 0, j] + r) * dphi(k[0, 0, j])
        return out

    right = dk_with(False, alpha)
    assert np.max(np.abs(right - fd[1][0, 0])) < 1e-6
    for wrong in (dk_with(True, alpha), dk_with(False, 1.0)):
        assert np.max(np.abs(wrong - fd[1][0, 0])) > 1e-3
