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
