"""Tensor-core backward (bf16, dk = dv = 64, causal and non-causal) vs the
fp64 oracle.

Shapes span one token, one partial chunk, exact chunk boundaries, a ragged
tail, segments of one and of several chunks (the segment plan depends on B*H
and N), so that both sweeps, the forward prefix scan and the reverse suffix
scan are all exercised; non-causal, the state pass over every segment and
passes A (dq, segment (R, r) records) and B (dk, dv from their total).
"""

import numpy as np
import pytest

import oracle as orc
import causal_linear_attention_la_gb300 as la
from causal_linear_attention_la_gb300 import synth
from helpers import build_lib, grad_errors, grad_tol, grads_ok, to_dev, to_host

TC_TOL = grad_tol("bf16", True)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_lib()
    la.lib()
    la.la_set_path(la.LA_PATH_AUTO)
    yield
    la.la_set_path(la.LA_PATH_AUTO)


def _grads(B, H, N, seed, eps=1e-6, causal=True):
    import torch
    q, k, v = synth.qkv(B, H, N, 64, 64, seed=seed, dtype="bf16")
    g = synth.upstream_grad(B, H, N, 64, seed=seed, dtype="bf16")
    got = la.backward(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"),
                      to_dev(g, "bf16"), causal=causal, eps=eps)
    torch.cuda.synchronize()
    want = orc.backward_recurrent(q, k, v, g, causal=causal, eps=eps)
    return got, want


def test_backward_path_is_tensor_core():
    assert la.la_backward_path(64, 64, la.LA_BF16, True) == 1
    assert la.la_backward_path(64, 64, la.LA_BF16, False) == 1
    assert la.la_backward_path(64, 64, la.LA_F32, True) == 0
    assert la.la_backward_path(128, 128, la.LA_BF16, True) == 0


@pytest.mark.parametrize("B,H,N", [
    (1, 1, 1),        # single token
    (1, 1, 100),      # one partial chunk
    (1, 1, 128),      # exactly one chunk
    (2, 1, 129),      # one chunk plus one token
    (1, 2, 300),      # ragged, one segment per chunk
    (1, 1, 4096),     # 32 one-chunk segments: long scans
    (4, 8, 1000),     # segments of two chunks, ragged last segment
    (2, 16, 3000),    # segments of six chunks
])
def test_backward_tensor_core(B, H, N):
    n0 = la.la_launch_count()
    got, want = _grads(B, H, N, seed=900 + N + B * H)
    # segment sums (only with more than one segment), sweep 1, sweep 2
    assert la.la_launch_count() - n0 in (2, 3)
    assert la.la_device_status(True) == la.LA_OK
    errs = grad_errors(got, want)
    assert grads_ok(errs, TC_TOL), errs


@pytest.mark.parametrize("B,H,N", [
    (1, 1, 1),        # single token
    (1, 1, 100),      # one partial chunk
    (2, 1, 129),      # one chunk plus one token
    (1, 2, 300),      # ragged, one segment per chunk
    (1, 1, 4096),     # 32 one-chunk segments: 32 records in every total
    (4, 8, 1000),     # segments of two chunks, ragged last segment
    (2, 16, 3000),    # segments of six chunks
])
def test_backward_tensor_core_noncausal(B, H, N):
    n0 = la.la_launch_count()
    got, want = _grads(B, H, N, seed=1900 + N + B * H, causal=False)
    # state pass, pass A, pass B
    assert la.la_launch_count() - n0 == 3
    assert la.la_device_status(True) == la.LA_OK
    errs = grad_errors(got, want)
    assert grads_ok(errs, TC_TOL), errs


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed", range(20))
def test_backward_tensor_core_seed_sweep(seed, causal):
    """Twenty seeds per form across the chunk and segment structure (a chunk
    and one token, ragged segments, many segments): every gradient within
    the bf16 bound of 2e-2 of its largest oracle magnitude."""
    N = (129, 1000, 4096, 8192)[seed % 4]
    got, want = _grads(1, 2, N, seed=7000 + seed, causal=causal)
    assert la.la_device_status(True) == la.LA_OK
    errs = grad_errors(got, want)
    assert grads_ok(errs, TC_TOL), errs


@pytest.mark.parametrize("causal", [True, False])
def test_backward_tensor_core_matches_cuda_core(causal):
    """Both paths implement the same gradient; on the same bf16 inputs they
    agree to the bf16 tolerance (each is also checked against the oracle)."""
    import torch
    B, H, N = 2, 4, 777
    q, k, v = synth.qkv(B, H, N, 64, 64, seed=31, dtype="bf16")
    g = synth.upstream_grad(B, H, N, 64, seed=31, dtype="bf16")
    args = [to_dev(x, "bf16") for x in (q, k, v, g)]
    tc = [t.clone() for t in la.backward(*args, causal=causal)]
    la.la_set_path(la.LA_PATH_SIMT)
    try:
        simt = [to_host(t) for t in la.backward(*args, causal=causal)]
        torch.cuda.synchronize()
    finally:
        la.la_set_path(la.LA_PATH_AUTO)
    errs = grad_errors(tc, simt)
    assert grads_ok(errs, TC_TOL), errs


@pytest.mark.parametrize("causal", [True, False])
def test_backward_tensor_core_eps_zero(causal):
    """eps = 0 is allowed; phi > 0 keeps every denominator positive."""
    got, want = _grads(1, 2, 513, seed=4242, eps=0.0, causal=causal)
    assert la.la_device_status(True) == la.LA_OK
    errs = grad_errors(got, want)
    assert grads_ok(errs, TC_TOL), errs


@pytest.mark.parametrize("causal", [True, False])
def test_backward_tensor_core_extreme_inputs(causal):
    """bf16 q, k of large magnitude (N(0, 30^2) clipped to +-100, so phi runs
    from e^-100 to 101) and eps = 0: finite gradients within the bf16 bound."""
    rng = np.random.default_rng(77 + causal)
    B, H, N = 1, 2, 700
    q = synth.round_to_bf16(np.clip(rng.standard_normal((B, H, N, 64)) * 30, -100, 100).astype(np.float32))
    k = synth.round_to_bf16(np.clip(rng.standard_normal((B, H, N, 64)) * 30, -100, 100).astype(np.float32))
    v = synth.round_to_bf16((rng.standard_normal((B, H, N, 64)) / 8).astype(np.float32))
    g = synth.round_to_bf16(rng.standard_normal((B, H, N, 64)).astype(np.float32))
    got = la.backward(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), to_dev(g, "bf16"),
                      causal=causal, eps=0.0)
    want = orc.backward_recurrent(q, k, v, g, causal=causal, eps=0.0)
    assert la.la_device_status(True) == la.LA_OK
    assert all(np.all(np.isfinite(to_host(t))) for t in got)
    errs = grad_errors(got, want)
    assert grads_ok(errs, TC_TOL), errs


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,N", [
    (1, 1, 100),      # one segment: no records (causal)
    (2, 3, 1000),     # several segments, ragged tail
    (6, 10, 2048),    # the forward's state pass splits each segment in two parts
    (4, 8, 1000),
])
def test_backward_saved(B, H, N, causal):
    """la_backward_saved reads the forward's state records from its workspace
    (two launches, no state pass) and gives the oracle's gradients."""
    import torch
    seed = 2900 + N + B * H
    q, k, v = synth.qkv(B, H, N, 64, 64, seed=seed, dtype="bf16")
    g = synth.upstream_grad(B, H, N, 64, seed=seed, dtype="bf16")
    qd, kd, vd, gd = (to_dev(x, "bf16") for x in (q, k, v, g))
    ws = torch.empty(max(1, la.la_forward_workspace_size(B, H, N, 64, 64, causal, la.LA_BF16)),
                     dtype=torch.uint8, device="cuda")
    la.forward(qd, kd, vd, causal=causal, workspace=ws)
    n0 = la.la_launch_count()
    got = la.backward_saved(qd, kd, vd, gd, ws, causal=causal)
    torch.cuda.synchronize()
    assert la.la_launch_count() - n0 == 2
    assert la.la_device_status(True) == la.LA_OK
    want = orc.backward_recurrent(q, k, v, g, causal=causal, eps=1e-6)
    errs = grad_errors(got, want)
    assert grads_ok(errs, TC_TOL), errs
