"""fp64 CPU oracle for the two state-update variants the pages describe next to
linear attention. TEST INFRASTRUCTURE (same rules as the rest of ``oracle``).

Sources:
- [LA-order] "Linear Attention, 곱의 순서를 바꾸면 생기는 일" (donmain.dev),
  the paragraphs after section "요약에는 자리가 모자란다": decay gating multiplies
  the whole summary by alpha < 1 every step; the delta rule reads the summary
  with the key before writing and adds only the difference to the target value.
- [SSM-LA] "상태공간모델·선형 어텐션 — 어텐션의 O(N²) 대안", section 3
  "대가 — 상태의 기억 길이": h_t = a h_{t-1} + x_t, impulse response a^t,
  half-life and effective memory length ~ 1/(1-a) ("직접 재 보기 C").

Readings (where the pages stop short):
- Decay: "the summary" of normalised linear attention is the pair (S, z); both
  decay, so each output is the decayed-weight average
  o_t = sum_j alpha^(t-j) w_j v_j / (sum_j alpha^(t-j) w_j + eps).
- Delta rule: the pages apply it to already-transformed keys with unnormalised
  reads (the feature map is left out of the example); so does this oracle:
  S <- S + k (v - S^T k)^T, o = S^T q, with the vectors as given (feature
  "identity" by default).
"""

import numpy as np

from .la_oracle import FEATURE_MAPS, _as64


def decode_steps_decay(S, z, q, k, v, alpha, eps=1e-6, feature="elu1"):
    """T steps of decayed linear attention on a given state, one per token:

        S <- alpha S + phi(k) v^T,  z <- alpha z + phi(k),
        o  = phi(q)^T S / (phi(q)^T z + eps)

    alpha: scalar or array broadcastable to the leading (batch, head) axes
    (one factor per head). Shapes: S [..., dk, dv], z [..., dk],
    q, k [..., T, dk], v [..., T, dv]. Returns (S', z', out [..., T, dv]).
    With alpha = 1 this is oracle.decode_steps.
    """
    S, z, q, k, v = _as64(S, z, q, k, v)
    a = np.asarray(alpha, dtype=np.float64)
    phi = FEATURE_MAPS[feature][0]
    T = q.shape[-2]
    out = np.zeros(q.shape[:-1] + (v.shape[-1],))
    for t in range(T):
        fk, fq = phi(k[..., t, :]), phi(q[..., t, :])
        S = a[..., None, None] * S + fk[..., :, None] * v[..., t, None, :]
        z = a[..., None] * z + fk
        num = np.einsum("...c,...cm->...m", fq, S)
        den = np.einsum("...c,...c->...", fq, z) + eps
        out[..., t, :] = num / den[..., None]
    return S, z, out


def backward_decay(q, k, v, g, alpha, eps=1e-6, feature="elu1"):
    """Gradients (dq, dk, dv) of L = sum(g * out) for the decayed causal
    attention of decode_steps_decay run from the zero state over the whole
    sequence (alpha fixed, one factor per head).

    The pages give only the decayed recurrence; its gradient follows by the
    chain rule through it. With D_t = phi(q_t).z_t + eps, o_t = S_t^T phi(q_t) / D_t:

        a_t = g_t / D_t,  b_t = -(g_t . o_t) / D_t
        dphi(q_t) = S_t a_t + b_t z_t                       (decayed S_t, z_t)
        R_j = phi(q_j) a_j^T + alpha R_{j+1},  r_j = b_j phi(q_j) + alpha r_{j+1}
        dphi(k_j) = R_j v_j + r_j,  dv_j = R_j^T phi(k_j)

    (S_{t+1} = alpha S_t + ..., so the adjoint carried from t+1 to t is
    scaled by alpha). With alpha = 1 this is oracle.backward_recurrent.
    Shapes as backward_recurrent; alpha broadcastable to (B, H).
    """
    q, k, v, g = _as64(q, k, v, g)
    phi, dphi = FEATURE_MAPS[feature]
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    a = np.broadcast_to(np.asarray(alpha, dtype=np.float64), (B, H))
    fq, fk = phi(q), phi(k)
    S = np.zeros((B, H, dk, dv))
    z = np.zeros((B, H, dk))
    at = np.zeros((B, H, N, dv))
    bt = np.zeros((B, H, N))
    dfq = np.zeros((B, H, N, dk))
    for t in range(N):
        S = a[..., None, None] * S + np.einsum("bhc,bhm->bhcm", fk[:, :, t], v[:, :, t])
        z = a[..., None] * z + fk[:, :, t]
        D = np.einsum("bhc,bhc->bh", fq[:, :, t], z) + eps
        o = np.einsum("bhc,bhcm->bhm", fq[:, :, t], S) / D[..., None]
        at[:, :, t] = g[:, :, t] / D[..., None]
        bt[:, :, t] = -np.einsum("bhm,bhm->bh", g[:, :, t], o) / D
        dfq[:, :, t] = np.einsum("bhcm,bhm->bhc", S, at[:, :, t]) + bt[:, :, t][..., None] * z
    R = np.zeros((B, H, dk, dv))
    r = np.zeros((B, H, dk))
    dfk = np.zeros((B, H, N, dk))
    dvv = np.zeros((B, H, N, dv))
    for j in range(N - 1, -1, -1):
        R = a[..., None, None] * R + np.einsum("bhc,bhm->bhcm", fq[:, :, j], at[:, :, j])
        r = a[..., None] * r + bt[:, :, j][..., None] * fq[:, :, j]
        dfk[:, :, j] = np.einsum("bhcm,bhm->bhc", R, v[:, :, j]) + r
        dvv[:, :, j] = np.einsum("bhcm,bhc->bhm", R, fk[:, :, j])
    return dfq * dphi(q), dfk * dphi(k), dvv


def decode_steps_delta(S, q, k, v, feature="identity"):
    """T delta-rule steps on a given state, one per token: read the state with
    the key, add the key times the difference to the value, read with the query:

        u = S^T phi(k),  S <- S + phi(k) (v - u)^T,  o = S^T phi(q)

    Shapes: S [..., dk, dv], q, k [..., T, dk], v [..., T, dv].
    Returns (S', out [..., T, dv]).
    """
    S, q, k, v = _as64(S, q, k, v)
    phi = FEATURE_MAPS[feature][0]
    T = q.shape[-2]
    out = np.zeros(q.shape[:-1] + (v.shape[-1],))
    for t in range(T):
        fk, fq = phi(k[..., t, :]), phi(q[..., t, :])
        u = np.einsum("...c,...cm->...m", fk, S)
        S = S + fk[..., :, None] * (v[..., t, :] - u)[..., None, :]
        out[..., t, :] = np.einsum("...c,...cm->...m", fq, S)
    return S, out


def impulse_response(a, steps):
    """h_t of h_t = a h_{t-1} + x_t with x_0 = 1 and x_t = 0 after ([SSM-LA] section 3)."""
    h, out = 0.0, []
    for t in range(steps):
        h = a * h + (1.0 if t == 0 else 0.0)
        out.append(h)
    return np.array(out)


def half_life(a):
    """Smallest number of steps t >= 1 after which the impulse has fallen to
    half or less: a^t <= 1/2."""
    t, h = 0, 1.0
    while True:
        t += 1
        h *= a
        if h <= 0.5:
            return t
