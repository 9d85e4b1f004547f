"""Decay-gated and delta-rule decode, the chunked delta rule, and the state
copy: CUDA path (through the C ABI) vs the fp64 oracle."""

import json
import os

import numpy as np
import pytest

import oracle as orc
import causal_linear_attention_la_gb300 as la
from causal_linear_attention_la_gb300 import synth
from helpers import TOL, build_lib, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_lib()
    la.lib()
    yield


def _prefill_state(B, H, dk, dv, dtype, seed):
    q0, k0, v0 = synth.qkv(B, H, 24, dk, dv, seed=seed, dtype=dtype)
    _, S, z = orc.forward_recurrent(q0, k0, v0, return_state=True)
    return S.astype(np.float32), z.astype(np.float32)


SHAPES = [(1, 1, 3, 16, 16), (2, 3, 5, 32, 64), (2, 2, 16, 128, 128), (3, 1, 33, 128, 16),
          (2, 2, 7, 16, 128), (64, 32, 16, 128, 128)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,T,dk,dv", SHAPES)
def test_decay_tokens(B, H, T, dk, dv, dtype):
    import torch
    S_ref, z_ref = _prefill_state(B, H, dk, dv, dtype, seed=5 * dk + dv)
    alpha_h = np.random.default_rng(T + H).uniform(0.5, 1.0, H).astype(np.float32)
    S = torch.from_numpy(S_ref).cuda()
    z = torch.from_numpy(z_ref).cuda()
    q, k, v = synth.qkv(B, H, T, dk, dv, seed=700 + T, dtype=dtype)
    out = la.decode_steps_decay(S, z, to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                torch.from_numpy(alpha_h).cuda())
    torch.cuda.synchronize()
    S_w, z_w, o_w = orc.decode_steps_decay(S_ref, z_ref, q, k, v,
                                           alpha=alpha_h.astype(np.float64)[None, :])
    assert rel_err(to_host(out), o_w, np.abs(v).max()) <= TOL[dtype]
    # the tensor-core decode carries psi(k) and the decay weights as bf16
    # hi + lo pairs (about 16 bits): 1e-5 of max|S|, as the undecayed one
    tc = la.la_decode_path(dk, dv, la.LA_BF16 if dtype == "bf16" else la.LA_F32, T) == 1
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= (1e-5 if tc else 1e-6)
    assert rel_err(to_host(z), z_w, np.abs(z_w).max()) <= 1e-6


@pytest.mark.parametrize("B,H,T,lo,hi", [(1, 1, 2, 0.9, 0.9), (2, 3, 15, 0.5, 1.0), (2, 1, 17, 0.5, 0.99),
                                         (3, 2, 40, 0.05, 0.3), (64, 32, 16, 0.9, 0.999),
                                         (1, 2, 200, 1.0, 1.0)])
def test_decay_tokens_tensor_core(B, H, T, lo, hi):
    """The tensor-core multi-token decode with decay (bf16, d = 128): against
    the oracle's decayed steps and against the CUDA-core kernel on the same
    inputs; partial and many groups, strong decay (a down to 0.05) and a = 1."""
    import torch
    d = 128
    assert la.la_decode_path(d, d, la.LA_BF16, T) == 1
    S_ref, z_ref = _prefill_state(B, H, d, d, "bf16", seed=T + 3)
    alpha_h = np.linspace(lo, hi, H).astype(np.float32)
    q, k, v = synth.qkv(B, H, T, d, d, seed=900 + T, dtype="bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    al = torch.from_numpy(alpha_h).cuda()
    S, z = torch.from_numpy(S_ref).cuda(), torch.from_numpy(z_ref).cuda()
    out = la.decode_steps_decay(S, z, qd, kd, vd, al)
    la.la_set_path(la.LA_PATH_SIMT)
    try:
        S2, z2 = torch.from_numpy(S_ref).cuda(), torch.from_numpy(z_ref).cuda()
        out2 = la.decode_steps_decay(S2, z2, qd, kd, vd, al)
        torch.cuda.synchronize()
    finally:
        la.la_set_path(la.LA_PATH_AUTO)
    assert la.la_device_status(True) == la.LA_OK
    S_w, z_w, o_w = orc.decode_steps_decay(S_ref, z_ref, q, k, v, alpha=alpha_h.astype(np.float64)[None, :])
    vmax = np.abs(v).max()
    assert rel_err(to_host(out), o_w, vmax) <= TOL["bf16"]
    assert rel_err(to_host(out), to_host(out2), vmax) <= TOL["bf16"]
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= 1e-5
    assert rel_err(to_host(z), z_w, np.abs(z_w).max()) <= 1e-6
    if lo == hi == 1.0:
        # a = 1 is the undecayed tensor-core decode
        S3, z3 = torch.from_numpy(S_ref).cuda(), torch.from_numpy(z_ref).cuda()
        out3 = la.decode_steps(S3, z3, qd, kd, vd)
        torch.cuda.synchronize()
        assert rel_err(to_host(out), to_host(out3), vmax) <= 1e-2
        assert rel_err(to_host(S), to_host(S3), float(S3.abs().max())) <= 1e-5


def test_decay_one_matches_plain_decode():
    import torch
    B, H, T, dk, dv = 2, 4, 20, 64, 64
    S_ref, z_ref = _prefill_state(B, H, dk, dv, "bf16", seed=8)
    q, k, v = [to_dev(x, "bf16") for x in synth.qkv(B, H, T, dk, dv, seed=9, dtype="bf16")]
    S1, z1 = torch.from_numpy(S_ref).cuda(), torch.from_numpy(z_ref).cuda()
    S2, z2 = S1.clone(), z1.clone()
    o1 = la.decode_steps_decay(S1, z1, q, k, v, torch.ones(H, device="cuda"))
    o2 = la.decode_steps(S2, z2, q, k, v)
    torch.cuda.synchronize()
    assert rel_err(to_host(o1), to_host(o2), 1.0) <= 1e-6
    assert rel_err(to_host(S1), to_host(S2), float(S2.abs().max())) <= 1e-6


def test_delta_rule_page_example_on_gpu():
    """The worked example, embedded in dk = dv = 16 (zeros elsewhere):
    (5, 3) then key (0.6, 0.8) with value 10 -> (7.76, 6.68); reads 10 and 7.76."""
    import torch
    with open(os.path.join(GOLDEN, "la_order_delta_rule.json")) as f:
        g = json.load(f)
    S = torch.zeros(1, 1, 16, 16, device="cuda")
    keys = g["k"] + [g["write"]["k"]]
    vals = [x[0] for x in g["v"]] + [g["write"]["v"][0]]
    k = torch.zeros(1, 1, 3, 16, device="cuda")
    v = torch.zeros(1, 1, 3, 16, device="cuda")
    q = torch.zeros(1, 1, 3, 16, device="cuda")
    for t in range(3):
        k[0, 0, t, :2] = torch.tensor(keys[t])
        v[0, 0, t, 0] = vals[t]
        q[0, 0, t, :2] = torch.tensor(g["reads_after"]["queries"][0])
    out = la.decode_steps_delta(S, q, k, v)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_host(S)[0, 0, :2, 0], g["S_after"], rtol=0, atol=1e-5)
    assert abs(float(out[0, 0, 2, 0]) - g["reads_after"]["values"][0]) <= 1e-5
    q1 = torch.zeros(1, 1, 1, 16, device="cuda")
    q1[0, 0, 0, 0] = 1.0
    o1 = la.decode_steps_delta(S, q1, torch.zeros_like(q1), torch.zeros(1, 1, 1, 16, device="cuda"))
    torch.cuda.synchronize()
    assert abs(float(o1[0, 0, 0, 0]) - g["reads_after"]["values"][1]) <= 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,T,dk,dv", SHAPES)
def test_delta_tokens(B, H, T, dk, dv, dtype):
    """Random unit-norm keys (rounded to the input dtype) on a random state."""
    import torch
    rng = np.random.default_rng(dk * 7 + dv + T)
    S0 = rng.standard_normal((B, H, dk, dv)).astype(np.float32)
    q, k, v = synth.qkv(B, H, T, dk, dv, seed=300 + T, dtype=dtype)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    qd, kd, vd = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    q, k = to_host(qd), to_host(kd)            # the values the kernel sees
    S = torch.from_numpy(S0).cuda()
    out = la.decode_steps_delta(S, qd, kd, vd)
    torch.cuda.synchronize()
    S_w, o_w = orc.decode_steps_delta(S0, q, k, v)
    scale = max(np.abs(o_w).max(), np.abs(v).max())
    assert rel_err(to_host(out), o_w, scale) <= TOL[dtype]
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= 1e-5


@pytest.mark.parametrize("B,H,T", [(1, 1, 2), (2, 3, 15), (2, 1, 17), (3, 2, 40), (64, 32, 16), (1, 2, 200)])
def test_delta_tokens_tensor_core(B, H, T):
    """The tensor-core delta-rule decode (bf16, d = 128): against the oracle's
    token steps and against the CUDA-core kernel on the same inputs; partial
    and many groups of 16, unit-norm keys on a random state."""
    import torch
    d = 128
    assert la.la_decode_path(d, d, la.LA_BF16, T) == 1
    rng = np.random.default_rng(T + 31)
    S0 = rng.standard_normal((B, H, d, d)).astype(np.float32)
    q, k, v = synth.qkv(B, H, T, d, d, seed=1300 + T, dtype="bf16")
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    qd, kd, vd = to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16")
    q, k = to_host(qd), to_host(kd)
    S = torch.from_numpy(S0).cuda()
    out = la.decode_steps_delta(S, qd, kd, vd)
    la.la_set_path(la.LA_PATH_SIMT)
    try:
        S2 = torch.from_numpy(S0).cuda()
        out2 = la.decode_steps_delta(S2, qd, kd, vd)
        torch.cuda.synchronize()
    finally:
        la.la_set_path(la.LA_PATH_AUTO)
    assert la.la_device_status(True) == la.LA_OK
    S_w, o_w = orc.decode_steps_delta(S0, q, k, v)
    scale = max(np.abs(o_w).max(), np.abs(v).max())
    assert rel_err(to_host(out), o_w, scale) <= TOL["bf16"]
    assert rel_err(to_host(out), to_host(out2), scale) <= TOL["bf16"]
    # the state read carries S as bf16 hi + lo and U' likewise (about 16 bits)
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= 1e-5


def _unit_qkv(B, H, N, d, dtype, seed):
    """Unit-norm queries and keys rounded to the input dtype, and the values
    the kernel sees (host copies read back from the device tensors)."""
    q, k, v = synth.qkv(B, H, N, d, d, seed=seed, dtype=dtype)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    qd, kd, vd = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    return (qd, kd, vd), (to_host(qd), to_host(kd), to_host(vd))


# N spans one partial chunk, exact multiples of the 32-token chunk, ragged
# tails and many chunks; d covers every supported head size
DELTA_SHAPES = [(1, 1, 1, 16), (2, 3, 31, 32), (2, 2, 32, 64), (2, 2, 33, 64),
                (1, 2, 100, 128), (3, 1, 257, 16), (2, 4, 1000, 128), (4, 2, 513, 32)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,N,d", DELTA_SHAPES)
def test_forward_delta_chunked(B, H, N, d, dtype):
    """Chunked delta rule (triangular solve per chunk) against the oracle's
    token-by-token recurrence from a random state."""
    import torch
    S0 = np.random.default_rng(N * 3 + d).standard_normal((B, H, d, d)).astype(np.float32)
    (qd, kd, vd), (q, k, v) = _unit_qkv(B, H, N, d, dtype, seed=900 + N)
    S = torch.from_numpy(S0).cuda()
    out = la.forward_delta(S, qd, kd, vd)
    torch.cuda.synchronize()
    S_w, o_w = orc.decode_steps_delta(S0, q, k, v)
    scale = max(np.abs(o_w).max(), np.abs(v).max())
    assert rel_err(to_host(out), o_w, scale) <= TOL[dtype]
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= 1e-5


def test_forward_delta_many_heads_tensor_core():
    """bf16, d = 128 and at least 64 heads: la_forward_delta takes the
    tensor-core group kernel; every output and the final states against the
    oracle's token recurrence (ragged last group)."""
    import torch
    B, H, N, d = 4, 16, 300, 128
    S0 = np.random.default_rng(5).standard_normal((B, H, d, d)).astype(np.float32)
    (qd, kd, vd), (q, k, v) = _unit_qkv(B, H, N, d, "bf16", seed=55)
    S = torch.from_numpy(S0).cuda()
    out = la.forward_delta(S, qd, kd, vd)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    S_w, o_w = orc.decode_steps_delta(S0, q, k, v)
    scale = max(np.abs(o_w).max(), np.abs(v).max())
    assert rel_err(to_host(out), o_w, scale) <= TOL["bf16"]
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= 1e-5


def test_forward_delta_whole_heads_d128():
    """Thirty-two heads of 2048 tokens at d = 128 (fp32), every output
    against the oracle; the final states too."""
    import torch
    B, H, N, d = 2, 16, 2048, 128
    S0 = np.zeros((B, H, d, d), np.float32)
    (qd, kd, vd), (q, k, v) = _unit_qkv(B, H, N, d, "f32", seed=77)
    S = torch.from_numpy(S0).cuda()
    out = la.forward_delta(S, qd, kd, vd)
    torch.cuda.synchronize()
    S_w, o_w = orc.decode_steps_delta(S0, q, k, v)
    assert rel_err(to_host(out), o_w, np.abs(o_w).max()) <= TOL["f32"]
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= 1e-5


def test_forward_delta_matches_token_steps():
    """The chunked form and the token-by-token kernel compute the same
    recurrence; they differ only in rounding order."""
    import torch
    B, H, N, d = 2, 3, 200, 64
    S0 = torch.randn(B, H, d, d, generator=torch.Generator().manual_seed(3)).cuda()
    (qd, kd, vd), _ = _unit_qkv(B, H, N, d, "f32", seed=5)
    S1, S2 = S0.clone(), S0.clone()
    o1 = la.forward_delta(S1, qd, kd, vd)
    o2 = la.decode_steps_delta(S2, qd, kd, vd)
    torch.cuda.synchronize()
    assert rel_err(to_host(o1), to_host(o2), float(o2.abs().max())) <= 1e-5
    assert rel_err(to_host(S1), to_host(S2), float(S2.abs().max())) <= 1e-5


def test_forward_delta_page_example():
    """The worked example of the delta rule as one sequence of three tokens
    (two writes, then the write under key (0.6, 0.8)), embedded in d = 16."""
    import torch
    with open(os.path.join(GOLDEN, "la_order_delta_rule.json")) as f:
        g = json.load(f)
    keys = g["k"] + [g["write"]["k"]]
    vals = [x[0] for x in g["v"]] + [g["write"]["v"][0]]
    S = torch.zeros(1, 1, 16, 16, device="cuda")
    q = torch.zeros(1, 1, 3, 16, device="cuda")
    k = torch.zeros(1, 1, 3, 16, device="cuda")
    v = torch.zeros(1, 1, 3, 16, device="cuda")
    for t in range(3):
        k[0, 0, t, :2] = torch.tensor(keys[t])
        v[0, 0, t, 0] = vals[t]
        q[0, 0, t, :2] = torch.tensor(g["reads_after"]["queries"][0])
    out = la.forward_delta(S, q, k, v)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_host(S)[0, 0, :2, 0], g["S_after"], rtol=0, atol=1e-5)
    assert abs(float(out[0, 0, 2, 0]) - g["reads_after"]["values"][0]) <= 1e-5


def test_forward_delta_edges():
    """N = 0 leaves the state alone; dk != dv is refused."""
    import torch
    S = torch.randn(1, 2, 32, 32, device="cuda")
    S_before = S.clone()
    e = torch.empty(1, 2, 0, 32, device="cuda")
    la.forward_delta(S, e, e, e)
    torch.cuda.synchronize()
    assert torch.equal(S, S_before)
    S2 = torch.zeros(1, 1, 32, 64, device="cuda")
    q = torch.zeros(1, 1, 4, 32, device="cuda")
    with pytest.raises(la.LaError):
        la.forward_delta(S2, q, q, torch.zeros(1, 1, 4, 64, device="cuda"))


def test_state_snapshot_restore_round_trip():
    """Save a state, step it, put the copy back and repeat the same steps: the
    outputs and states repeat bit for bit; without z only S is copied."""
    import torch
    B, H, T, dk, dv = 4, 8, 9, 128, 64
    S_ref, z_ref = _prefill_state(B, H, dk, dv, "bf16", seed=12)
    S, z = torch.from_numpy(S_ref).cuda(), torch.from_numpy(z_ref).cuda()
    snapS, snapz = torch.empty_like(S), torch.empty_like(z)
    la.state_copy(snapS, S, snapz, z)
    q, k, v = [to_dev(x, "bf16") for x in synth.qkv(B, H, T, dk, dv, seed=13, dtype="bf16")]
    o1 = la.decode_steps(S, z, q, k, v)
    S1, z1 = S.clone(), z.clone()
    la.state_copy(S, snapS, z, snapz)
    torch.cuda.synchronize()
    assert torch.equal(S, torch.from_numpy(S_ref).cuda()) and torch.equal(z, torch.from_numpy(z_ref).cuda())
    o2 = la.decode_steps(S, z, q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S, S1) and torch.equal(z, z1)
    only = torch.zeros_like(S)
    la.state_copy(only, S)
    torch.cuda.synchronize()
    assert torch.equal(only, S)


# ---------------------------------------------------------------------------
# Decay-gated forward (chunked, tensor cores) vs the oracle recurrence
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("B,H,N", [
    (1, 1, 1),         # one token
    (1, 1, 100),       # one partial chunk
    (2, 1, 129),       # a chunk and one token
    (2, 3, 1000),      # several segments, ragged tail
    (1, 1, 4096),      # many one-chunk segments
    (6, 10, 2049),     # state pass in several parts per segment, one-token tail
])
def test_forward_decay(B, H, N):
    import torch
    from helpers import STATE_TOL, Z_TOL_DECAY_BF16
    q, k, v = synth.qkv(B, H, N, 64, 64, seed=40 + N + H, dtype="bf16")
    alpha_h = np.random.default_rng(N).uniform(0.5, 1.0, H).astype(np.float32)
    out, S, z = la.forward_decay(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"),
                                 torch.from_numpy(alpha_h).cuda(), return_state=True)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    S_w, z_w, o_w = orc.decode_steps_decay(np.zeros((B, H, 64, 64)), np.zeros((B, H, 64)), q, k, v,
                                           alpha=alpha_h.astype(np.float64)[None, :])
    err = rel_err(to_host(out), o_w, np.abs(v).max())
    assert err <= TOL["bf16"], err
    s_err = rel_err(to_host(S), S_w, np.abs(S_w).max())
    z_err = rel_err(to_host(z), z_w, np.abs(z_w).max())
    assert s_err <= STATE_TOL["bf16"] and z_err <= Z_TOL_DECAY_BF16, (s_err, z_err)


def test_forward_decay_one_is_forward():
    import torch
    B, H, N = 2, 4, 3000
    q, k, v = [to_dev(x, "bf16") for x in synth.qkv(B, H, N, 64, 64, seed=61, dtype="bf16")]
    o1 = la.forward_decay(q, k, v, torch.ones(H, device="cuda"))
    o2 = la.forward(q, k, v)
    torch.cuda.synchronize()
    # the same chunk loop; the plain forward's state records are centred
    # (psi = phi - 1 sums plus the value sums) and round differently from the
    # decayed records, so the outputs agree to within one bf16 step of
    # max|v| (2^-8), not bit for bit
    assert rel_err(to_host(o1), to_host(o2), float(v.abs().max())) <= 2.0 ** -8


# ---------------------------------------------------------------------------
# Decay-gated backward (CUDA-core sweeps with decayed segment records) vs the
# oracle's chain-rule gradient of the decayed recurrence
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,N,d", [
    (1, 1, 1, 64),       # one token
    (1, 2, 100, 64),     # one partial tile per sequence
    (2, 3, 1000, 64),    # several segments, ragged tail
    (1, 1, 4096, 16),    # many segments: long decayed scans
    (2, 2, 777, 128),
    (4, 8, 3000, 64),
])
def test_backward_decay(B, H, N, d, dtype):
    import torch
    from helpers import grad_errors, grad_tol, grads_ok
    q, k, v = synth.qkv(B, H, N, d, d, seed=70 + N + d, dtype=dtype)
    g = synth.upstream_grad(B, H, N, d, seed=70 + N + d, dtype=dtype)
    alpha_h = np.random.default_rng(N + H).uniform(0.5, 1.0, H).astype(np.float32)
    got = la.backward_decay(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), to_dev(g, dtype),
                            torch.from_numpy(alpha_h).cuda())
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    want = orc.backward_decay(q, k, v, g, alpha=alpha_h.astype(np.float64)[None, :])
    errs = grad_errors(got, want)
    assert grads_ok(errs, grad_tol(dtype, False)), errs


def test_backward_decay_one_is_backward():
    """alpha = 1 is the plain gradient: the same CUDA-core sweeps without decay."""
    import torch
    B, H, N, d = 2, 3, 1500, 64
    q, k, v = synth.qkv(B, H, N, d, d, seed=81, dtype="f32")
    g = synth.upstream_grad(B, H, N, d, seed=81, dtype="f32")
    args = [to_dev(x, "f32") for x in (q, k, v, g)]
    got = la.backward_decay(*args, torch.ones(H, device="cuda"))
    plain = la.backward(*args)
    torch.cuda.synchronize()
    for a, b in zip(got, plain):
        assert rel_err(to_host(a), to_host(b), float(b.abs().max())) <= 1e-6
