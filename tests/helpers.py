"""Shared test helpers: device transfer and the parity metrics."""

import numpy as np

# Tolerances (max abs error relative to max|V| for outputs, relative to the
# largest oracle gradient magnitude for gradients).
TOL = {"f32": 1e-4, "bf16": 2e-2}

# Final-state tolerance (max abs error relative to max|S|). With bf16 inputs
# the tensor cores multiply phi(k) rounded to bf16 (relative error up to
# 2^-9 per term); the sum of N such terms with random-sign values keeps a
# relative error near 2^-9 / sqrt(3) ~ 1e-3 (2.4e-3 observed at N = 32768),
# bounded here at 1e-2. fp32 inputs keep fp32 phi throughout.
STATE_TOL = {"f32": 1e-5, "bf16": 1e-2}

# Normaliser tolerance (max abs error relative to max z). With bf16 inputs at
# d = 64 the tensor cores sum z from the same bf16-rounded phi(k) that feed S
# (so S and z weight every token alike): each term carries a relative error
# of at most half a bf16 ulp, 2^-8, which is the bound at N = 1 (2.8e-3
# observed); over N terms the unbiased rounding errors shrink like 1/sqrt(N).
# Bounded like the state, at 1e-2.
Z_TOL = {"f32": 1e-5, "bf16": 1e-2}

# Gradient tolerances of the tensor-core backward (bf16 operands, fp32
# accumulation), per gradient, max abs error relative to that gradient's
# largest oracle magnitude. dq is ill-conditioned in the phi values: dphi(q_t)
# = sum_j phi(k_j) ((v_j - o_t) . a_t), whose terms are 10-50 times the sum for
# random inputs, so the bf16 rounding of phi(k) in the intra-chunk contraction
# dP' phi(K) (relative 2^-9 per term) and of a and dP' leaves ~2.5 % (median)
# and up to 5.9 % (worst of 80 seeds and shapes, causal and not, N = 129 ..
# 4096) of max|dq|; an fp64 emulation of the kernel's roundings reproduces the
# GPU's figure to three digits. dk and dv stay below 1.3 %. The CUDA-core path
# (fp32 arithmetic) keeps TOL.
GRAD_TOL_TC = {"dq": 8e-2, "dk": 2e-2, "dv": 2e-2}


def grad_tol(dtype, tensor_core):
    """Per-gradient tolerances (dq, dk, dv) for a backward path."""
    if tensor_core and dtype == "bf16":
        return [GRAD_TOL_TC[n] for n in ("dq", "dk", "dv")]
    return [TOL[dtype]] * 3


def grads_ok(errs, tols):
    return all(e <= t for e, t in zip(errs, tols))


def torch_dtype(name):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def to_dev(x, dtype):
    """float32 host array holding values of ``dtype`` -> exact CUDA tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(torch_dtype(dtype))


def to_host(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def rel_err(got, want, scale):
    return float(np.max(np.abs(np.asarray(got, np.float64) - want)) / scale)


def build_lib():
    from causal_linear_attention_la_gb300.build import build
    return build()


def grad_errors(got, want):
    """Per-tensor max abs error of (dq, dk, dv), each relative to that tensor's
    largest oracle magnitude, floored at 1e-2 x the largest magnitude of all
    three: for very short sequences dq and dk shrink to O(eps) by cancellation
    (a single token's output is v_0 s / (s + eps)), and a relative error of a
    vanishing quantity says nothing about the arithmetic."""
    want = [np.asarray(w, np.float64) for w in want]
    floor = 1e-2 * max(float(np.abs(w).max()) for w in want)
    out = []
    for a, b in zip(got, want):
        out.append(rel_err(to_host(a), b, max(float(np.abs(b).max()), floor)))
    return out
