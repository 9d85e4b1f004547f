"""Decode and backward parity: CUDA path (through the C ABI) vs the fp64 oracle."""

import numpy as np
import pytest

import oracle as orc
import causal_linear_attention_la_gb300 as la
from causal_linear_attention_la_gb300 import synth
from helpers import TOL, build_lib, grad_errors, grad_tol, grads_ok, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_lib()
    la.lib()
    yield
    la.la_set_path(la.LA_PATH_AUTO)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,dk,dv", [(1, 1, 16, 16), (2, 3, 32, 64),
                                       (4, 2, 128, 128), (3, 1, 128, 16),
                                       (2, 2, 16, 128), (64, 32, 128, 128)])
def test_decode_steps(B, H, dk, dv, dtype):
    import torch
    # start from the oracle state of a short prefill, then step
    N0 = 40
    q0, k0, v0 = synth.qkv(B, H, N0, dk, dv, seed=dk + dv, dtype=dtype)
    _, S_ref, z_ref = orc.forward_recurrent(q0, k0, v0, return_state=True)
    S = torch.from_numpy(S_ref.astype(np.float32)).cuda()
    z = torch.from_numpy(z_ref.astype(np.float32)).cuda()
    S_ref, z_ref = S_ref.astype(np.float32).astype(np.float64), z_ref.astype(np.float32).astype(np.float64)
    for step in range(3):
        q, k, v = synth.decode_token(B, H, dk, dv, seed=7, step=step, dtype=dtype)
        out = la.decode_step(S, z, to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
        torch.cuda.synchronize()
        S_ref, z_ref, o_ref = orc.decode_step(S_ref, z_ref, q, k, v)
        err = rel_err(to_host(out), o_ref, np.abs(v).max())
        assert err <= TOL[dtype], (step, err)
        assert rel_err(to_host(S), S_ref, np.abs(S_ref).max()) <= 1e-6
        assert rel_err(to_host(z), z_ref, np.abs(z_ref).max()) <= 1e-6


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,T,dk,dv", [(1, 1, 2, 16, 16), (2, 3, 5, 32, 64),
                                         (4, 2, 16, 128, 128), (3, 1, 33, 128, 16),
                                         (2, 2, 7, 16, 128), (1, 2, 64, 64, 64),
                                         (64, 32, 16, 128, 128)])
def test_decode_tokens(B, H, T, dk, dv, dtype):
    """T tokens per call (la_decode_steps) from a prefill state vs the oracle's
    T single steps: outputs, and the state after the call."""
    import torch
    N0 = 24
    q0, k0, v0 = synth.qkv(B, H, N0, dk, dv, seed=3 * dk + dv, dtype=dtype)
    _, S_ref, z_ref = orc.forward_recurrent(q0, k0, v0, return_state=True)
    S_ref, z_ref = S_ref.astype(np.float32), z_ref.astype(np.float32)
    S = torch.from_numpy(S_ref).cuda()
    z = torch.from_numpy(z_ref).cuda()
    q, k, v = synth.qkv(B, H, T, dk, dv, seed=900 + T, dtype=dtype)
    out = la.decode_steps(S, z, to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
    torch.cuda.synchronize()
    S_w, z_w, o_w = orc.decode_steps(S_ref, z_ref, q, k, v)
    assert la.la_device_status(True) == la.LA_OK
    err = rel_err(to_host(out), o_w, np.abs(v).max())
    assert err <= TOL[dtype], err
    # the tensor-core kernel (bf16, d = 128) updates the state through MMAs
    # whose psi(k) operand is split into two bf16 parts (about 16 bits):
    # 1e-5 of max|S|; the CUDA-core kernels update in fp32 FMAs
    s_tol = 1e-5 if la.la_decode_path(dk, dv, la.LA_BF16 if dtype == "bf16" else la.LA_F32, T) == 1 else 1e-6
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= s_tol
    assert rel_err(to_host(z), z_w, np.abs(z_w).max()) <= 1e-6


@pytest.mark.parametrize("B,H,T", [(1, 1, 2), (2, 3, 15), (1, 2, 16), (2, 1, 17), (3, 2, 40),
                                   (64, 32, 16), (1, 1, 200)])
def test_decode_tokens_tensor_core(B, H, T):
    """The tensor-core multi-token decode (bf16, d = 128) against the oracle's
    T single steps and against the CUDA-core kernel on the same inputs:
    groups of 16 tokens, partial last groups, one and many groups."""
    import torch
    d = 128
    assert la.la_decode_path(d, d, la.LA_BF16, T) == 1
    q0, k0, v0 = synth.qkv(B, H, 40, d, d, seed=T + 7, dtype="bf16")
    _, S_ref, z_ref = orc.forward_recurrent(q0, k0, v0, return_state=True)
    S_ref, z_ref = S_ref.astype(np.float32), z_ref.astype(np.float32)
    q, k, v = synth.qkv(B, H, T, d, d, seed=500 + T, dtype="bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    S, z = torch.from_numpy(S_ref).cuda(), torch.from_numpy(z_ref).cuda()
    out = la.decode_steps(S, z, qd, kd, vd)
    la.la_set_path(la.LA_PATH_SIMT)
    try:
        assert la.la_decode_path(d, d, la.LA_BF16, T) == 0
        S2, z2 = torch.from_numpy(S_ref).cuda(), torch.from_numpy(z_ref).cuda()
        out2 = la.decode_steps(S2, z2, qd, kd, vd)
        torch.cuda.synchronize()
    finally:
        la.la_set_path(la.LA_PATH_AUTO)
    assert la.la_device_status(True) == la.LA_OK
    S_w, z_w, o_w = orc.decode_steps(S_ref, z_ref, q, k, v)
    vmax = np.abs(v).max()
    assert rel_err(to_host(out), o_w, vmax) <= TOL["bf16"]
    assert rel_err(to_host(out), to_host(out2), vmax) <= TOL["bf16"]
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= 1e-5
    assert rel_err(to_host(z), z_w, np.abs(z_w).max()) <= 1e-6


def test_decode_tokens_tensor_core_extreme_inputs():
    """bf16 q, k of large magnitude (|x| up to 100) and eps = 0 through the
    tensor-core decode: finite outputs within the bf16 bound."""
    import torch
    rng = np.random.default_rng(91)
    B, H, T, d = 2, 2, 20, 128
    mk = lambda s: synth.round_to_bf16(np.clip(rng.standard_normal((B, H, T, d)) * s, -100, 100).astype(np.float32))
    q, k = mk(30.0), mk(30.0)
    v = synth.round_to_bf16((rng.standard_normal((B, H, T, d)) / 8).astype(np.float32))
    S0 = np.zeros((B, H, d, d), np.float32)
    z0 = np.zeros((B, H, d), np.float32)
    S, z = torch.from_numpy(S0).cuda(), torch.from_numpy(z0).cuda()
    out = la.decode_steps(S, z, to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), eps=0.0)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    _, _, o_w = orc.decode_steps(S0, z0, q, k, v, eps=0.0)
    got = to_host(out)
    assert np.all(np.isfinite(got))
    assert rel_err(got, o_w, np.abs(v).max()) <= TOL["bf16"]


def test_decode_tokens_edge_cases():
    """T = 0 leaves the state untouched; T = 1 is la_decode_step bit for bit."""
    import torch
    B, H, dk, dv = 2, 3, 64, 32
    S0 = torch.randn(B, H, dk, dv, device="cuda").abs()
    z0 = torch.randn(B, H, dk, device="cuda").abs() + 1.0
    S, z = S0.clone(), z0.clone()
    e = torch.empty(B, H, 0, dk, device="cuda", dtype=torch.bfloat16)
    out = la.decode_steps(S, z, e, e, torch.empty(B, H, 0, dv, device="cuda", dtype=torch.bfloat16))
    torch.cuda.synchronize()
    assert out.shape == (B, H, 0, dv)
    assert torch.equal(S, S0) and torch.equal(z, z0)
    q, k, v = synth.qkv(B, H, 1, dk, dv, seed=77, dtype="bf16")
    S1, z1 = S0.clone(), z0.clone()
    o1 = la.decode_steps(S1, z1, to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"))
    S2, z2 = S0.clone(), z0.clone()
    o2 = la.decode_step(S2, z2, to_dev(q[:, :, 0], "bf16"), to_dev(k[:, :, 0], "bf16"),
                        to_dev(v[:, :, 0], "bf16"))
    torch.cuda.synchronize()
    assert torch.equal(o1[:, :, 0], o2) and torch.equal(S1, S2) and torch.equal(z1, z2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_then_decode_matches_forward(dtype):
    import torch
    B, H, N, dk, dv = 2, 2, 300, 64, 64
    q, k, v = synth.qkv(B, H, N + 1, dk, dv, seed=31, dtype=dtype)
    full = orc.forward_recurrent(q, k, v)
    _, S, z = la.forward(to_dev(q[:, :, :N], dtype), to_dev(k[:, :, :N], dtype),
                         to_dev(v[:, :, :N], dtype), return_state=True)
    out = la.decode_step(S, z, to_dev(q[:, :, N], dtype), to_dev(k[:, :, N], dtype),
                         to_dev(v[:, :, N], dtype))
    torch.cuda.synchronize()
    assert rel_err(to_host(out), full[:, :, N], np.abs(v).max()) <= TOL[dtype]


PATHS = [la.LA_PATH_AUTO, la.LA_PATH_SIMT]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,N,dk,dv", [
    (1, 1, 1, 16, 16),
    (1, 1, 64, 16, 16),
    (2, 1, 129, 64, 64),
    (1, 2, 700, 32, 128),
    (1, 1, 1500, 128, 128),
    (2, 3, 333, 128, 128),
    (1, 2, 2049, 128, 128),
    (1, 3, 333, 128, 16),
])
def test_backward_shapes(B, H, N, dk, dv, causal, dtype, path):
    import torch
    seed = 500 + N + dk
    q, k, v = synth.qkv(B, H, N, dk, dv, seed=seed, dtype=dtype)
    g = synth.upstream_grad(B, H, N, dv, seed=seed, dtype=dtype)
    want = orc.backward_recurrent(q, k, v, g, causal=causal, eps=1e-6)
    la.la_set_path(path)
    try:
        tc = la.la_backward_path(dk, dv, la.LA_BF16 if dtype == "bf16" else la.LA_F32, causal) == 1
        got = la.backward(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                          to_dev(g, dtype), causal=causal, eps=1e-6)
        torch.cuda.synchronize()
    finally:
        la.la_set_path(la.LA_PATH_AUTO)
    errs = grad_errors(got, want)
    assert grads_ok(errs, grad_tol(dtype, tc)), errs
