"""Shared test helpers: device transfer and the parity metrics."""

import numpy as np

# Tolerances (max abs error relative to max|V| for outputs, relative to the
# largest oracle gradient magnitude for gradients).
TOL = {"f32": 1e-4, "bf16": 2e-2}


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
