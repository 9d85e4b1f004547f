"""The error model behind the tensor-core backward's dq bound, on the CPU.

The tensor-core sweep computes dq from bf16-rounded operands: phi(q) and
phi(k), the row-scaled gradient a = g / D, the bf16 copy of the chunk's
starting state S, and the packed dP' = (a V^T + b) masked, with fp32 (here
fp64) accumulation. This file restates those roundings over the oracle's
inputs (the chunked form of the gradient with chunks of 128 tokens) and
checks two facts the bound rests on:

* the modelled roundings give a dq error of a few percent of max|dq| for
  random inputs (0.0261 for the inputs of the smoke check, which the GPU
  reproduces to three digits), while the model without roundings matches the
  oracle to fp64 precision;
* the rounding of phi(k) in the intra-chunk contraction dP' phi(K) is the
  largest single source: with that one operand exact (everything else still
  rounded as the kernels do) the error falls by a third to a half.
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


def _dq_model(q, k, v, g, rounded=True, exact_phik_intra=False, eps=1e-6):
    """dq of the causal chunked gradient with the tensor-core roundings."""
    rd = _bf16 if rounded else (lambda x: np.asarray(x, np.float64))
    B, H, N, d = q.shape
    dq = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            Q, K, V, G = (x[b, h].astype(np.float64) for x in (q, k, v, g))
            pq, pk, pk_exact = rd(_phi(Q)), rd(_phi(K)), _phi(K)
            S = np.zeros((d, d))
            z = np.zeros(d)
            for c0 in range(0, N, C):
                sl = slice(c0, min(N, c0 + C))
                P = np.tril(pq[sl] @ pk[sl].T)
                Sb = rd(S)
                O = pq[sl] @ Sb + rd(P) @ V[sl]
                den = P.sum(1) + pq[sl] @ z + eps
                a = rd(G[sl] / den[:, None])
                bb = -(G[sl] * O).sum(1) / den ** 2
                dPp = rd(np.tril(a @ V[sl].T + bb[:, None]))
                kin = pk_exact[sl] if exact_phik_intra else pk[sl]
                dQ = a @ Sb.T + dPp @ kin + bb[:, None] * z[None, :]
                dq[b, h, sl] = dQ * np.minimum(pq[sl], 1.0)
                S = S + pk[sl].T @ V[sl]
                z = z + pk[sl].sum(0)
    return dq


def _rel(x, want):
    return float(np.abs(x - want).max() / np.abs(want).max())


def _inputs(seed, B=1, H=2, N=300, d=64):
    q, k, v = synth.qkv(B, H, N, d, d, seed=seed, dtype="bf16")
    g = synth.upstream_grad(B, H, N, d, seed=seed, dtype="bf16")
    return q, k, v, g


def test_model_without_rounding_is_the_oracle():
    q, k, v, g = _inputs(7)
    want = orc.backward_recurrent(q, k, v, g)[0]
    assert _rel(_dq_model(q, k, v, g, rounded=False), want) < 1e-10


@pytest.mark.parametrize("seed", [11, 13])
def test_rounding_model_error_and_its_source(seed):
    q, k, v, g = _inputs(seed)
    want = orc.backward_recurrent(q, k, v, g)[0]
    full = _rel(_dq_model(q, k, v, g), want)
    assert 0.015 < full < 0.06, full          # a few percent of max|dq|
    if seed == 11:                            # the smoke check's inputs
        assert abs(full - 0.0261) < 5e-4, full
    exact_intra = _rel(_dq_model(q, k, v, g, exact_phik_intra=True), want)
    assert exact_intra < 0.75 * full, (full, exact_intra)
