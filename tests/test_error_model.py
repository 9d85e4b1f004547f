"""Why the tensor-core backward centres phi(k), on the CPU.

dq is ill-conditioned in the feature values: dphi(q_t) = sum_j phi(k_j)
((v_j - o_t) . a_t), and phi(k) = 1 + psi(k) has a common part (the 1) whose
terms cancel almost exactly ("Transformers are RNNs" review, section
"그래디언트 계산 — 선형 시간·상수 메모리", gives the cumulative-sum method; the
formulas are derived from the forward definition). This file restates the
tensor-core sweep's arithmetic over the oracle's inputs, chunks of 128 tokens,
in two forms:

* plain: phi(q), phi(k), a = g / D, the bf16 copy of the chunk's starting
  state and the packed dP' = (a V^T + b) masked are rounded to bf16, with
  fp32 (here fp64) accumulation;
* centred (what the kernels do): the tensor cores see psi(k) = phi(k) - 1 in
  place of phi(k), the state and z are carried as their psi sums, and the
  parts that hold the 1 (the row sum s_t of phi(q_t), the value sums V_t and
  the token count) are exact scalars per row; b_t is formed from the rounded
  a_t that the MMAs read, and the intra-chunk dP' = dP + b enters as the
  separately rounded pair [dP | b].

It checks that both models reproduce the oracle exactly without rounding,
that the plain form's rounding costs percents of max|dq| for random inputs,
and that the centred form stays far inside the 2e-2 bound.
"""

import numpy as np
import pytest

import oracle as orc
from causal_linear_attention_la_gb300 import synth

C = 128


def _bf16(x):
    """Round to bf16 (nearest even) and back."""
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _dq_model(q, k, v, g, centred, rounded=True, eps=1e-6):
    """dq of the causal chunked gradient with the tensor-core roundings."""
    rd = _bf16 if rounded else (lambda x: np.asarray(x, np.float64))
    B, H, N, d = q.shape
    dq = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            Q, K, V, G = (x[b, h].astype(np.float64) for x in (q, k, v, g))
            pq = rd(_phi(Q))
            kin = rd(_phi(K) - 1.0) if centred else rd(_phi(K))
            S = np.zeros((d, d))
            z = np.zeros(d)
            vsum = np.zeros(d)
            n = 0
            for c0 in range(0, N, C):
                sl = slice(c0, min(N, c0 + C))
                m = sl.stop - sl.start
                P = np.tril(pq[sl] @ kin[sl].T)
                Sb = rd(S)
                O = pq[sl] @ Sb + rd(P) @ V[sl]
                if centred:
                    s = pq[sl].sum(1)
                    nt = n + np.arange(1, m + 1)
                    den = s * nt + P.sum(1) + pq[sl] @ z + eps
                    a = rd(G[sl] / den[:, None])
                    dP = a @ V[sl].T
                    av = a @ vsum + np.tril(dP).sum(1)          # a_t . V_t
                    bb = -(s * av + (a * O).sum(1)) / den
                    cc = av + nt * bb
                    # dP and b packed separately: [dP | b] [psiK ; psiK]
                    dPp = rd(np.tril(dP)) + rd(bb)[:, None] * np.tril(np.ones((m, m)))
                    dQ = a @ Sb.T + dPp @ kin[sl] + bb[:, None] * z[None, :] + cc[:, None]
                else:
                    den = P.sum(1) + pq[sl] @ z + eps
                    a = rd(G[sl] / den[:, None])
                    bb = -(G[sl] * O).sum(1) / den ** 2
                    dPp = rd(np.tril(a @ V[sl].T + bb[:, None]))
                    dQ = a @ Sb.T + dPp @ kin[sl] + bb[:, None] * z[None, :]
                dq[b, h, sl] = dQ * np.minimum(pq[sl], 1.0)
                S = S + kin[sl].T @ V[sl]
                # z from the exact fp32 sums (the kernels' column sums)
                z = z + ((_phi(K[sl]) - 1.0) if centred else kin[sl]).sum(0)
                vsum = vsum + V[sl].sum(0)
                n += m
    return dq


def _rel(x, want):
    return float(np.abs(x - want).max() / np.abs(want).max())


def _inputs(seed, B=1, H=2, N=300, d=64):
    q, k, v = synth.qkv(B, H, N, d, d, seed=seed, dtype="bf16")
    g = synth.upstream_grad(B, H, N, d, seed=seed, dtype="bf16")
    return q, k, v, g


@pytest.mark.parametrize("centred", [False, True])
def test_model_without_rounding_is_the_oracle(centred):
    q, k, v, g = _inputs(7)
    want = orc.backward_recurrent(q, k, v, g)[0]
    assert _rel(_dq_model(q, k, v, g, centred, rounded=False), want) < 1e-10


def test_centring_removes_the_cancellation_error():
    plain, centred = [], []
    for seed in (11, 13, 1, 2, 3, 4):
        q, k, v, g = _inputs(seed)
        want = orc.backward_recurrent(q, k, v, g)[0]
        plain.append(_rel(_dq_model(q, k, v, g, False), want))
        centred.append(_rel(_dq_model(q, k, v, g, True), want))
    # the plain form: percents of max|dq|, beyond the 2e-2 bound for some inputs
    assert max(plain) > 2e-2 and min(plain) > 1e-2, plain
    # the centred form: well inside the bound, several times smaller
    assert max(centred) < 1e-2, centred
    assert all(c < p / 3 for c, p in zip(centred, plain)), (plain, centred)
