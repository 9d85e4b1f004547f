"""Plain fp64 oracle: what causal linear attention computes, written out.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline). Not on the
product path; it imports nothing from the product package.

Sources, cited by page title and section / equation / figure:

* [LA-state] "Linear Attention: KV를 고정 크기 상태에 누적하기"
  (ai-systems-engineering.com) -- the state S, the normaliser z, the
  index convention (S_{t+1} includes token t) and the 3-token worked example.
* [LA-order] "Linear Attention, 곱의 순서를 바꾸면 생기는 일" (donmain.dev) --
  the association reorder and the scalar-value worked example.
* [RNN-review] "Transformers are RNNs" paper review (taepoung.github.io,
  Jump2Paper archive) -- phi(x) = elu(x) + 1, the causal cumulative sums
  S_i, z_i and the RNN form with s_0 = 0, z_0 = 0.
* [SSM-LA] "상태공간모델·선형 어텐션 — 어텐션의 O(N²) 대안" -- section 2,
  the masked O(N^2) form written next to the recurrence.

Conventions (all arrays float64, layout [B, H, N, d]):
  q, k : [B, H, N, dk]  raw (pre feature map) queries / keys
  v    : [B, H, N, dv]  values (the feature map is never applied to v)
  out  : [B, H, N, dv]
  S    : [B, H, dk, dv] rows = key components, columns = value components
  z    : [B, H, dk]

Readings where the pages are silent:
  * eps is added to the denominator: o = phi(q)^T S / (phi(q)^T z + eps).
  * no 1/sqrt(d) scale inside the linear form.
  * causal means j <= t inclusive: output t reads the state that already
    holds token t.
  * gradients: the pages lost the formulas; ``backward_recurrent`` and
    ``backward_masked`` are two independent derivations from the forward
    definition, pinned by finite differences in the tests.

parity: every function here is pinned by a test in tests/test_oracle.py.
"""

from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# Feature maps
# ----------------------------------------------------------------------------


def elu(x):
    """ELU with alpha = 1: x for x >= 0, exp(x) - 1 for x < 0.

    [RNN-review], feature-map table ("x>=0 이면 x, x<0 이면 exp(x)-1").
    """
    x = np.asarray(x, dtype=np.float64)
    return np.where(x >= 0.0, x, np.expm1(np.minimum(x, 0.0)))


def phi_elu1(x):
    """phi(x) = elu(x) + 1, applied elementwise, to q and to k separately.

    [RNN-review], feature-map table (the "+1" offset keeps it non-negative);
    [LA-state], section "Softmax를 바꾸는 이유" (ELU(x)+1 from the paper's 3.2).

    For x < 0, elu(x) + 1 = (exp(x) - 1) + 1 = exp(x) in real arithmetic; it is
    evaluated as exp(x) so that it stays positive where exp(x) < 2^-53 (the
    literal sum would round to 0 there). The tests check that both forms agree
    to one unit of 1.0 everywhere.
    """
    x = np.asarray(x, dtype=np.float64)
    return np.where(x >= 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def phi_elu1_prime(x):
    """d phi / dx: 1 for x >= 0, exp(x) for x < 0 (derivative of expm1)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x >= 0.0, 1.0, np.exp(np.minimum(x, 0.0)))


def phi_identity(x):
    """phi(x) = x. [LA-state] and [LA-order] run their worked examples on
    already-transformed vectors, i.e. with the feature map left out."""
    return np.asarray(x, dtype=np.float64)


def _identity_prime(x):
    return np.ones_like(np.asarray(x, dtype=np.float64))


FEATURE_MAPS = {
    "elu1": (phi_elu1, phi_elu1_prime),
    "identity": (phi_identity, _identity_prime),
}


def _as64(*arrays):
    return [np.asarray(a, dtype=np.float64) for a in arrays]


# ----------------------------------------------------------------------------
# Forward: the masked O(N^2) form
# ----------------------------------------------------------------------------


def forward_masked(q, k, v, causal=True, eps=1e-6, feature="elu1",
                   normalise=True):
    """Masked quadratic form.

    o_t = sum_{j<=t} (phi(q_t).phi(k_j)) v_j / (sum_{j<=t} phi(q_t).phi(k_j) + eps)

    [SSM-LA] section 2, left-hand side of the equation; non-causal: the sum runs
    over every j ([RNN-review], generalised attention with sim = phi(q)^T phi(k)).
    With ``normalise=False`` returns the numerator alone, i.e. the
    "(Q~ K~^T) V" product of [LA-state] section "KV부터 계산하면 줄어드는 것".
    """
    q, k, v = _as64(q, k, v)
    phi = FEATURE_MAPS[feature][0]
    fq, fk = phi(q), phi(k)
    scores = np.einsum("bhtc,bhjc->bhtj", fq, fk)          # sim(q_t, k_j)
    if causal:
        n = scores.shape[-1]
        scores = scores * np.tril(np.ones((n, n)))         # keep j <= t
    num = np.einsum("bhtj,bhjm->bhtm", scores, v)
    if not normalise:
        return num
    den = scores.sum(axis=-1) + eps
    return num / den[..., None]


# ----------------------------------------------------------------------------
# Forward: the recurrence
# ----------------------------------------------------------------------------


def forward_recurrent(q, k, v, causal=True, eps=1e-6, feature="elu1",
                      normalise=True, return_state=False):
    """Token-by-token recurrence on the fixed-size state.

    S_0 = 0, z_0 = 0;  S_{t+1} = S_t + phi(k_t) v_t^T;  z_{t+1} = z_t + phi(k_t);
    y_t^T = phi(q_t)^T S_{t+1} / (phi(q_t)^T z_{t+1} + eps).

    [LA-state] section "상태 갱신과 읽기를 식으로 정리하기" (the three equations);
    [RNN-review] RNN-form table (s_0 = 0, z_0 = 0).  Non-causal: every query
    reads the full-sequence state S_N = K~^T V ([LA-state], fig. 2 bottom).

    Returns out, or (out, S_N, z_N) when ``return_state``.
    """
    q, k, v = _as64(q, k, v)
    phi = FEATURE_MAPS[feature][0]
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, dk, dv))
    z = np.zeros((B, H, dk))
    out = np.zeros((B, H, N, dv))

    def read(fq_t):
        num = np.einsum("bhc,bhcm->bhm", fq_t, S)
        if not normalise:
            return num
        den = np.einsum("bhc,bhc->bh", fq_t, z) + eps
        return num / den[..., None]

    if causal:
        for t in range(N):
            fk_t = phi(k[:, :, t, :])
            S = S + np.einsum("bhc,bhm->bhcm", fk_t, v[:, :, t, :])
            z = z + fk_t
            out[:, :, t, :] = read(phi(q[:, :, t, :]))
    else:
        for t in range(N):
            fk_t = phi(k[:, :, t, :])
            S = S + np.einsum("bhc,bhm->bhcm", fk_t, v[:, :, t, :])
            z = z + fk_t
        for t in range(N):
            out[:, :, t, :] = read(phi(q[:, :, t, :]))
    if return_state:
        return out, S, z
    return out


def decode_step(S, z, q, k, v, eps=1e-6, feature="elu1"):
    """One recurrent inference step on a given state, inclusive of the token.

    S' = S + phi(k) v^T; z' = z + phi(k); o = phi(q)^T S' / (phi(q)^T z' + eps).

    [LA-state] section "상태 갱신과 읽기를 식으로 정리하기";
    [LA-order] section "곱의 순서를 바꾸면 기억이 요약이 된다" (add the outer
    product to the summary, then read it with the query).
    Shapes: S [..., dk, dv], z [..., dk], q,k [..., dk], v [..., dv].
    Returns (S', z', o); the inputs are not modified.
    """
    S, z, q, k, v = _as64(S, z, q, k, v)
    phi = FEATURE_MAPS[feature][0]
    fk, fq = phi(k), phi(q)
    S_new = S + fk[..., :, None] * v[..., None, :]
    z_new = z + fk
    num = np.einsum("...c,...cm->...m", fq, S_new)
    den = np.einsum("...c,...c->...", fq, z_new) + eps
    return S_new, z_new, num / den[..., None]


def decode_steps(S, z, q, k, v, eps=1e-6, feature="elu1"):
    """T consecutive recurrent steps on a given state, one per token.

    The step of decode_step applied to tokens 0 .. T-1 in order (the
    recurrence of [LA-state] section "상태 갱신과 읽기를 식으로 정리하기",
    started from (S, z) instead of zero).
    Shapes: S [..., dk, dv], z [..., dk], q,k [..., T, dk], v [..., T, dv].
    Returns (S', z', out [..., T, dv]); the inputs are not modified.
    """
    S, z, q, k, v = _as64(S, z, q, k, v)
    T = q.shape[-2]
    out = np.zeros(q.shape[:-1] + (v.shape[-1],))
    for t in range(T):
        S, z, out[..., t, :] = decode_step(S, z, q[..., t, :], k[..., t, :], v[..., t, :],
                                           eps=eps, feature=feature)
    return S, z, out


def output_at(q_bh, k_bh, v_bh, t, causal=True, eps=1e-6, feature="elu1"):
    """Output of one query position of one (batch, head), by the definition.

    o_t = sum_j w_j v_j / (sum_j w_j + eps), w_j = phi(q_t).phi(k_j), j <= t
    (all j when not causal). [SSM-LA] section 2. Used to check single
    sampled outputs of large problems without running the whole recurrence.
    q_bh, k_bh: [N, dk]; v_bh: [N, dv].
    """
    q_bh, k_bh, v_bh = _as64(q_bh, k_bh, v_bh)
    phi = FEATURE_MAPS[feature][0]
    last = t + 1 if causal else q_bh.shape[0]
    w = phi(k_bh[:last]) @ phi(q_bh[t])
    return (w @ v_bh[:last]) / (w.sum() + eps)


# ----------------------------------------------------------------------------
# Backward
# ----------------------------------------------------------------------------
#
# [RNN-review] section "그래디언트 계산 — 선형 시간·상수 메모리" states that the
# gradient is written as cumulative sums so no per-token state is stored; its
# formulas did not survive extraction. Derivation from the forward definition,
# with g_t = dL/do_t, D_t = phi(q_t).z_t + eps and o_t = n_t / D_t:
#   a_t = g_t / D_t                       (dL/dn_t)
#   b_t = -(g_t . o_t) / D_t              (dL/dD_t)
#   dphi(q_t) = S_t a_t + b_t z_t         (S_t, z_t inclusive of token t)
#   R_j = sum_{t>=j} phi(q_t) a_t^T,  r_j = sum_{t>=j} b_t phi(q_t)
#   dphi(k_j) = R_j v_j + r_j,        dv_j = R_j^T phi(k_j)
#   dq = dphi(q) * phi'(q),           dk = dphi(k) * phi'(k)
# Non-causal: S_t -> S_N, z_t -> z_N, R_j -> R_0, r_j -> r_0.


def backward_recurrent(q, k, v, g, causal=True, eps=1e-6, feature="elu1"):
    """Gradients by forward and reverse cumulative sums (see block comment).

    Returns (dq, dk, dv) for the scalar loss L = sum(g * out).
    """
    q, k, v, g = _as64(q, k, v, g)
    phi, dphi = FEATURE_MAPS[feature]
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    fq, fk = phi(q), phi(k)

    # forward sweep: states S_t, z_t inclusive of token t (or S_N, z_N)
    S = np.zeros((B, H, dk, dv))
    z = np.zeros((B, H, dk))
    if not causal:
        S = np.einsum("bhtc,bhtm->bhcm", fk, v)
        z = fk.sum(axis=2)
    a = np.zeros((B, H, N, dv))
    bsc = np.zeros((B, H, N))
    dfq = np.zeros((B, H, N, dk))
    for t in range(N):
        if causal:
            S = S + np.einsum("bhc,bhm->bhcm", fk[:, :, t], v[:, :, t])
            z = z + fk[:, :, t]
        num = np.einsum("bhc,bhcm->bhm", fq[:, :, t], S)
        D = np.einsum("bhc,bhc->bh", fq[:, :, t], z) + eps
        o = num / D[..., None]
        a[:, :, t] = g[:, :, t] / D[..., None]
        bsc[:, :, t] = -np.einsum("bhm,bhm->bh", g[:, :, t], o) / D
        dfq[:, :, t] = (np.einsum("bhcm,bhm->bhc", S, a[:, :, t])
                        + bsc[:, :, t][..., None] * z)

    # reverse sweep: R_j, r_j inclusive of token j (or R_0, r_0)
    R = np.zeros((B, H, dk, dv))
    r = np.zeros((B, H, dk))
    if not causal:
        R = np.einsum("bhtc,bhtm->bhcm", fq, a)
        r = np.einsum("bht,bhtc->bhc", bsc, fq)
    dfk = np.zeros((B, H, N, dk))
    dvv = np.zeros((B, H, N, dv))
    for j in range(N - 1, -1, -1):
        if causal:
            R = R + np.einsum("bhc,bhm->bhcm", fq[:, :, j], a[:, :, j])
            r = r + bsc[:, :, j][..., None] * fq[:, :, j]
        dfk[:, :, j] = np.einsum("bhcm,bhm->bhc", R, v[:, :, j]) + r
        dvv[:, :, j] = np.einsum("bhcm,bhc->bhm", R, fk[:, :, j])
    return dfq * dphi(q), dfk * dphi(k), dvv


def backward_masked(q, k, v, g, causal=True, eps=1e-6, feature="elu1"):
    """Gradients of the masked O(N^2) form by the matrix chain rule.

    With W = (phi(Q) phi(K)^T) masked, n = W V, D = W 1 + eps, o = n / D:
      dL/dW_tj = a_t . v_j + b_t  (kept where the mask is 1)
      dphi(Q) = dW phi(K);  dphi(K) = dW^T phi(Q);  dV = W^T A
    An independent second path to the same gradients.
    """
    q, k, v, g = _as64(q, k, v, g)
    phi, dphi = FEATURE_MAPS[feature]
    N = q.shape[2]
    fq, fk = phi(q), phi(k)
    mask = np.tril(np.ones((N, N))) if causal else np.ones((N, N))
    W = np.einsum("bhtc,bhjc->bhtj", fq, fk) * mask
    num = np.einsum("bhtj,bhjm->bhtm", W, v)
    D = W.sum(axis=-1) + eps
    o = num / D[..., None]
    A = g / D[..., None]
    bsc = -np.einsum("bhtm,bhtm->bht", g, o) / D
    dW = (np.einsum("bhtm,bhjm->bhtj", A, v) + bsc[..., None]) * mask
    dfq = np.einsum("bhtj,bhjc->bhtc", dW, fk)
    dfk = np.einsum("bhtj,bhtc->bhjc", dW, fq)
    dvv = np.einsum("bhtj,bhtm->bhjm", W, A)
    return dfq * dphi(q), dfk * dphi(k), dvv


def loss_dot(q, k, v, g, causal=True, eps=1e-6, feature="elu1"):
    """L = sum(g * out) with out from the masked form; the scalar whose
    gradients the two backward functions return (used by finite differences)."""
    out = forward_masked(q, k, v, causal=causal, eps=eps, feature=feature)
    return float(np.sum(np.asarray(g, dtype=np.float64) * out))
