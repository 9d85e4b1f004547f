"""Pins for the fp64 oracle: page values, closed forms, invariants, brute force.

Nothing here touches the GPU or the CUDA library. Each pin is chosen so that a
plausible mistake in the oracle (a dropped term, an exclusive instead of an
inclusive state, a transposed outer product, a wrong feature-map branch, a
sign error in a gradient) fails at least one of them; the last block plants
such mistakes in copies of oracle functions and checks that the pins catch them.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle as orc
from causal_linear_attention_la_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bh(x):
    """[N, d] -> [1, 1, N, d]"""
    return np.asarray(x, dtype=np.float64)[None, None]


# ---------------------------------------------------------------------------
# Worked example of "Linear Attention: KV를 고정 크기 상태에 누적하기", figs. 2-6
# ---------------------------------------------------------------------------


def check_three_token_example(recurrent=orc.forward_recurrent,
                              masked=orc.forward_masked,
                              decode=orc.decode_step):
    g = _load("la_state_three_tokens.json")
    q, k, v = _bh(g["q"]), _bh(g["k"]), _bh(g["v"])
    # fig. 4: S_1, S_2, S_3 after one, two, three tokens
    for n, key in ((1, "S1"), (2, "S2"), (3, "S3")):
        _, S, _ = recurrent(q[:, :, :n], k[:, :, :n], v[:, :, :n],
                            feature="identity", normalise=False,
                            return_state=True)
        np.testing.assert_array_equal(S[0, 0], np.array(g["states"][key], float))
    # fig. 6: z_3 = [2, 1]
    _, _, z = recurrent(q, k, v, feature="identity", return_state=True)
    np.testing.assert_array_equal(z[0, 0], np.array(g["normaliser"]["z3"], float))
    # fig. 5: reads of S_3 = weighted sums over the three tokens
    qs = _bh(g["reads_of_S3"]["queries"])
    reads = masked(qs, k, v, causal=False, feature="identity", normalise=False)
    np.testing.assert_array_equal(reads[0, 0],
                                  np.array(g["reads_of_S3"]["values"], float))
    # fig. 2 bottom: both association orders give Q~ S_3 before normalisation
    full_m = masked(q, k, v, causal=False, feature="identity", normalise=False)
    full_r = recurrent(q, k, v, causal=False, feature="identity",
                       normalise=False)
    want = np.array(g["full_sequence_unnormalised"]["value"], float)
    np.testing.assert_array_equal(full_m[0, 0], want)
    np.testing.assert_array_equal(full_r[0, 0], want)
    # fig. 6: causal output of p2 = [3,1] / 2 = [1.5, 0.5] (eps = 0)
    num = recurrent(q, k, v, feature="identity", normalise=False)
    np.testing.assert_array_equal(num[0, 0, 2], np.array(g["normaliser"]["num_q2"], float))
    y = recurrent(q, k, v, feature="identity", eps=0.0)
    np.testing.assert_array_equal(y[0, 0, 2], np.array(g["normaliser"]["y2"], float))
    y_m = masked(q, k, v, feature="identity", eps=0.0)
    np.testing.assert_array_equal(y_m[0, 0, 2], np.array(g["normaliser"]["y2"], float))
    # the same convention gives y_0 = v_0 and y_1 = v_1 (one non-zero score each)
    np.testing.assert_array_equal(y[0, 0, 0], [2.0, 0.0])
    np.testing.assert_array_equal(y[0, 0, 1], [0.0, 3.0])
    # fig. 3 and the [0.3, 0.7] example: one outer product from the zero state
    S0, z0 = np.zeros((2, 2)), np.zeros(2)
    S1, _, _ = decode(S0, z0, np.array([1.0, 0.0]), np.array(g["k"][2], float),
                      np.array(g["v"][2], float), feature="identity")
    np.testing.assert_array_equal(S1, np.array(g["outer_p2"]["value"], float))
    ex = g["outer_extra"]
    S1, _, _ = decode(S0, z0, np.array([1.0, 0.0]), np.array(ex["k"]),
                      np.array(ex["v"], float), feature="identity")
    np.testing.assert_allclose(S1, np.array(ex["value"]), rtol=0, atol=1e-15)


def test_three_token_example():
    check_three_token_example()


# ---------------------------------------------------------------------------
# Scalar-value example of "Linear Attention, 곱의 순서를 바꾸면 생기는 일"
# ---------------------------------------------------------------------------


def check_scalar_value_example(recurrent=orc.forward_recurrent,
                               masked=orc.forward_masked):
    g = _load("la_order_scalar_value.json")
    k2, v2 = _bh(g["k"]), _bh(g["v"])
    _, S, _ = recurrent(k2, k2, v2, feature="identity", normalise=False,
                        return_state=True)
    np.testing.assert_array_equal(S[0, 0, :, 0], np.array(g["S_after_two"], float))
    qs = _bh(g["reads_after_two"]["queries"])
    reads = masked(qs, k2, v2, causal=False, feature="identity", normalise=False)
    np.testing.assert_array_equal(reads[0, 0, :, 0], g["reads_after_two"]["values"])
    k3 = _bh(g["k"] + [g["third"]["k"]])
    v3 = _bh(g["v"] + [g["third"]["v"]])
    _, S, _ = recurrent(k3, k3, v3, feature="identity", normalise=False,
                        return_state=True)
    np.testing.assert_allclose(S[0, 0, :, 0], g["third"]["S_after"], rtol=0, atol=1e-12)
    qs = _bh(g["third"]["reads"]["queries"])
    reads = masked(qs, k3, v3, causal=False, feature="identity", normalise=False)
    np.testing.assert_allclose(reads[0, 0, :, 0], g["third"]["reads"]["values"],
                               rtol=0, atol=1e-12)


def test_scalar_value_example():
    check_scalar_value_example()


# ---------------------------------------------------------------------------
# Feature map: closed form
# ---------------------------------------------------------------------------


def test_phi_closed_form():
    xs = [-700.0, -30.0, -2.5, -1e-8, 0.0, 1e-8, 0.5, 3.0, 1e6]
    for x in xs:
        want = x + 1.0 if x >= 0 else math.exp(x)
        got = float(orc.phi_elu1(x))
        assert got == pytest.approx(want, rel=1e-15, abs=0.0), x
        dwant = 1.0 if x >= 0 else math.exp(x)
        assert float(orc.phi_elu1_prime(x)) == pytest.approx(dwant, rel=1e-15)
    assert float(orc.phi_elu1(0.0)) == 1.0
    # the literal elu(x) + 1 agrees to within rounding of the "+1"
    xw = np.linspace(-60, 60, 20001)
    np.testing.assert_allclose(orc.phi_elu1(xw), orc.elu(xw) + 1.0, rtol=0, atol=2.3e-16)
    x = np.linspace(-50, 50, 100001)
    assert np.all(orc.phi_elu1(x) > 0)
    # derivative agrees with a central difference away from the kink
    xx = np.array([-3.0, -0.7, -0.01, 0.01, 0.9, 4.0])
    h = 1e-6
    fd = (orc.phi_elu1(xx + h) - orc.phi_elu1(xx - h)) / (2 * h)
    np.testing.assert_allclose(orc.phi_elu1_prime(xx), fd, rtol=1e-8)


# ---------------------------------------------------------------------------
# Equivalences and invariants on seeded inputs
# ---------------------------------------------------------------------------


def _rand(B=2, H=2, N=19, dk=5, dv=3, seed=7):
    q, k, v = synth.qkv(B, H, N, dk, dv, seed, dtype="f32")
    return [np.asarray(a, np.float64) for a in (q, k, v)]


@pytest.mark.parametrize("causal", [True, False])
def test_masked_equals_recurrent(causal):
    q, k, v = _rand()
    a = orc.forward_masked(q, k, v, causal=causal)
    b = orc.forward_recurrent(q, k, v, causal=causal)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_convex_hull():
    q, k, v = _rand(N=40, seed=11)
    for eps in (0.0, 1e-6, 0.5):
        o = orc.forward_recurrent(q, k, v, eps=eps)
        for t in range(q.shape[2]):
            lo = v[:, :, : t + 1].min(axis=2)
            hi = v[:, :, : t + 1].max(axis=2)
            if eps > 0:
                lo, hi = np.minimum(lo, 0), np.maximum(hi, 0)
            assert np.all(o[:, :, t] >= lo - 1e-12)
            assert np.all(o[:, :, t] <= hi + 1e-12)


def test_equal_keys_prefix_mean():
    rng = np.random.default_rng(3)
    N, dk, dv, eps = 12, 4, 3, 0.25
    kk = rng.standard_normal(dk)
    k = np.tile(kk, (N, 1))[None, None]
    q = rng.standard_normal((1, 1, N, dk))
    v = rng.standard_normal((1, 1, N, dv))
    o = orc.forward_recurrent(q, k, v, eps=eps)
    for t in range(N):
        s = float(orc.phi_elu1(q[0, 0, t]) @ orc.phi_elu1(kk))
        D = (t + 1) * s
        want = v[0, 0, : t + 1].mean(axis=0) * D / (D + eps)
        np.testing.assert_allclose(o[0, 0, t], want, rtol=1e-13)


def test_single_token():
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((3, 1, 1, 1, 6))
    eps = 0.3
    o = orc.forward_recurrent(q, k, v[..., :4], eps=eps)
    s = float(orc.phi_elu1(q[0, 0, 0]) @ orc.phi_elu1(k[0, 0, 0]))
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0, :4] * s / (s + eps), rtol=1e-14)


def test_noncausal_last_row_and_state():
    q, k, v = _rand(B=1, H=1, N=9, dk=3, dv=2, seed=2)
    oc = orc.forward_recurrent(q, k, v, causal=True)
    on = orc.forward_recurrent(q, k, v, causal=False)
    np.testing.assert_allclose(on[:, :, -1], oc[:, :, -1], rtol=1e-14)
    _, S, z = orc.forward_recurrent(q, k, v, causal=False, return_state=True)
    # S_N = phi(K)^T V written as plain Python loops
    fk = orc.phi_elu1(k[0, 0])
    for c in range(3):
        for m in range(2):
            acc = 0.0
            for t in range(9):
                acc += fk[t, c] * v[0, 0, t, m]
            assert S[0, 0, c, m] == pytest.approx(acc, rel=1e-14)
        assert z[0, 0, c] == pytest.approx(sum(fk[t, c] for t in range(9)), rel=1e-14)


def test_output_at_matches_forward():
    q, k, v = _rand(B=1, H=2, N=17, seed=9)
    for causal in (True, False):
        o = orc.forward_masked(q, k, v, causal=causal)
        for h in range(2):
            for t in (0, 5, 16):
                got = orc.output_at(q[0, h], k[0, h], v[0, h], t, causal=causal)
                np.testing.assert_allclose(got, o[0, h, t], rtol=1e-13)


def test_decode_continues_prefill():
    q, k, v = _rand(B=2, H=3, N=14, dk=4, dv=5, seed=4)
    full = orc.forward_recurrent(q, k, v)
    for t in (0, 1, 7, 13):
        _, S, z = orc.forward_recurrent(q[:, :, :t], k[:, :, :t], v[:, :, :t],
                                        return_state=True)
        S2, z2, o = orc.decode_step(S, z, q[:, :, t], k[:, :, t], v[:, :, t])
        np.testing.assert_allclose(o, full[:, :, t], rtol=1e-13, atol=1e-15)
        _, S_ref, z_ref = orc.forward_recurrent(q[:, :, : t + 1], k[:, :, : t + 1],
                                                v[:, :, : t + 1], return_state=True)
        np.testing.assert_allclose(S2, S_ref, rtol=1e-14)
        np.testing.assert_allclose(z2, z_ref, rtol=1e-14)


def test_decode_two_steps_on_page_example():
    g = _load("la_state_three_tokens.json")
    S, z = np.zeros((2, 2)), np.zeros(2)
    outs = []
    for t in range(3):
        S, z, o = orc.decode_step(S, z, np.array(g["q"][t], float),
                                  np.array(g["k"][t], float),
                                  np.array(g["v"][t], float),
                                  eps=0.0, feature="identity")
        outs.append(o)
    np.testing.assert_array_equal(S, np.array(g["states"]["S3"], float))
    np.testing.assert_array_equal(outs[2], np.array(g["normaliser"]["y2"], float))


def test_decode_steps_on_page_example():
    """Three tokens in one multi-token call from the zero state reproduce the
    worked example's S_3 (fig. 4) and its outputs (fig. 6: y_2 = [1.5, 0.5])."""
    g = _load("la_state_three_tokens.json")
    S, z, out = orc.decode_steps(np.zeros((2, 2)), np.zeros(2),
                                 np.array(g["q"], float), np.array(g["k"], float),
                                 np.array(g["v"], float), eps=0.0, feature="identity")
    np.testing.assert_array_equal(S, np.array(g["states"]["S3"], float))
    np.testing.assert_array_equal(z, np.array(g["normaliser"]["z3"], float))
    np.testing.assert_array_equal(out[0], [2.0, 0.0])
    np.testing.assert_array_equal(out[1], [0.0, 3.0])
    np.testing.assert_array_equal(out[2], np.array(g["normaliser"]["y2"], float))


def test_decode_steps_continue_prefill():
    """From the state of a prefill of t tokens, T steps give the whole-sequence
    outputs t .. t+T-1 and the state of the first t+T tokens; T = 0 changes
    nothing."""
    q, k, v = _rand(B=2, H=2, N=20, dk=4, dv=3, seed=12)
    full, S_all, z_all = orc.forward_recurrent(q, k, v, return_state=True)
    for t, T in ((0, 20), (5, 1), (7, 9), (19, 1)):
        _, S, z = orc.forward_recurrent(q[:, :, :t], k[:, :, :t], v[:, :, :t],
                                        return_state=True)
        S2, z2, out = orc.decode_steps(S, z, q[:, :, t:t + T], k[:, :, t:t + T],
                                       v[:, :, t:t + T])
        np.testing.assert_allclose(out, full[:, :, t:t + T], rtol=1e-12, atol=1e-14)
        _, S_ref, z_ref = orc.forward_recurrent(q[:, :, :t + T], k[:, :, :t + T],
                                                v[:, :, :t + T], return_state=True)
        np.testing.assert_allclose(S2, S_ref, rtol=1e-13)
        np.testing.assert_allclose(z2, z_ref, rtol=1e-13)
    S0, z0 = S_all.copy(), z_all.copy()
    S1, z1, out = orc.decode_steps(S0, z0, q[:, :, :0], k[:, :, :0], v[:, :, :0])
    assert out.shape == (2, 2, 0, 3)
    np.testing.assert_array_equal(S1, S_all)
    np.testing.assert_array_equal(z1, z_all)


# ---------------------------------------------------------------------------
# Backward: finite differences (brute force) and the two derivations
# ---------------------------------------------------------------------------


def _fd_grads(q, k, v, g, causal, eps, h=1e-6):
    grads = []
    for which in range(3):
        arrs = [q.copy(), k.copy(), v.copy()]
        x = arrs[which]
        d = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = orc.loss_dot(*arrs, g, causal=causal, eps=eps)
            x[idx] = old - h
            lm = orc.loss_dot(*arrs, g, causal=causal, eps=eps)
            x[idx] = old
            d[idx] = (lp - lm) / (2 * h)
        grads.append(d)
    return grads


@pytest.mark.parametrize("causal", [True, False])
def test_backward_finite_differences(causal):
    rng = np.random.default_rng(17 + causal)
    B, H, N, dk, dv = 1, 2, 7, 3, 4
    q = rng.standard_normal((B, H, N, dk))
    k = rng.standard_normal((B, H, N, dk))
    v = rng.standard_normal((B, H, N, dv))
    g = rng.standard_normal((B, H, N, dv))
    eps = 0.05
    fd = _fd_grads(q, k, v, g, causal, eps)
    for fn in (orc.backward_recurrent, orc.backward_masked):
        got = fn(q, k, v, g, causal=causal, eps=eps)
        for a, b in zip(got, fd):
            err = np.max(np.abs(a - b)) / np.max(np.abs(b))
            assert err < 1e-6, (fn.__name__, err)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_two_derivations_agree(causal):
    q, k, v = _rand(B=2, H=2, N=33, dk=6, dv=5, seed=21)
    g = synth.upstream_grad(2, 2, 33, 5, 21, dtype="f32").astype(np.float64)
    a = orc.backward_recurrent(q, k, v, g, causal=causal)
    b = orc.backward_masked(q, k, v, g, causal=causal)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-11 * np.max(np.abs(y)))


# ---------------------------------------------------------------------------
# The pins catch planted mistakes (mutants are copies made here, on the CPU)
# ---------------------------------------------------------------------------


def _mutant_recurrent_exclusive(q, k, v, causal=True, eps=1e-6, feature="elu1",
                                normalise=True, return_state=False):
    # reads the state before adding token t (an off-by-one in the index)
    q, k, v = [np.asarray(a, np.float64) for a in (q, k, v)]
    phi = orc.FEATURE_MAPS[feature][0]
    B, H, N, dk = q.shape
    S = np.zeros((B, H, dk, v.shape[-1]))
    z = np.zeros((B, H, dk))
    out = np.zeros(v.shape)
    for t in range(N):
        fq = phi(q[:, :, t])
        num = np.einsum("bhc,bhcm->bhm", fq, S)
        den = np.einsum("bhc,bhc->bh", fq, z) + eps
        out[:, :, t] = num if not normalise else num / np.where(den == 0, 1, den)[..., None]
        fk = phi(k[:, :, t])
        S = S + np.einsum("bhc,bhm->bhcm", fk, v[:, :, t])
        z = z + fk
    return (out, S, z) if return_state else out


def _mutant_recurrent_transposed(q, k, v, causal=True, eps=1e-6, feature="elu1",
                                 normalise=True, return_state=False):
    # stores v k^T instead of k v^T (only shape-compatible when dk == dv)
    res = orc.forward_recurrent(q, k, v, causal, eps, feature, normalise, True)
    out, S, z = res
    S = np.swapaxes(S, -1, -2)
    return (out, S, z) if return_state else out


def test_pins_catch_planted_mistakes():
    with pytest.raises(AssertionError):
        check_three_token_example(recurrent=_mutant_recurrent_exclusive)
    with pytest.raises(AssertionError):
        check_three_token_example(recurrent=_mutant_recurrent_transposed)
    # a feature map without the +1 offset is not positive
    x = np.linspace(-5, 5, 11)
    assert not np.all(orc.elu(x) > 0)
    # a backward with the normaliser term dropped fails finite differences
    rng = np.random.default_rng(1)
    q, k, v, g = rng.standard_normal((4, 1, 1, 5, 3))
    fd = _fd_grads(q, k, v, g, True, 0.05)
    dq, _, _ = orc.backward_recurrent(q, k, v, g, eps=0.05)
    # the b_t z_t term of dphi(q) is the normaliser's share of the gradient
    fq = orc.phi_elu1(q)
    D = np.cumsum(orc.phi_elu1(k), axis=2)
    o = orc.forward_recurrent(q, k, v, eps=0.05)
    Dt = np.einsum("bhtc,bhtc->bht", fq, D) + 0.05
    b = -np.einsum("bhtm,bhtm->bht", g, o) / Dt
    dq_wrong = dq - (b[..., None] * D) * orc.phi_elu1_prime(q)
    assert np.max(np.abs(dq - fd[0])) < 1e-6
    assert np.max(np.abs(dq_wrong - fd[0])) > 1e-3


# ---------------------------------------------------------------------------
# Input generator (no method arithmetic): bf16 rounding is round-nearest-even
# ---------------------------------------------------------------------------


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = synth.normal((4096,), seed=123, scale=3.0, dtype="f32")
    x = np.concatenate([x, np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 0.0],
                                    np.float32)])
    ours = synth.round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_synth_is_deterministic():
    a = synth.qkv(1, 2, 8, 4, 4, seed=3)
    b = synth.qkv(1, 2, 8, 4, 4, seed=3)
    c = synth.qkv(1, 2, 8, 4, 4, seed=4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a[0], c[0])
    assert not np.array_equal(a[0], a[1])
