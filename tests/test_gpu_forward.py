"""Forward parity: CUDA path (through the C ABI) vs the fp64 oracle.

Errors are max |out_gpu - out_oracle| / max|V| over the whole tensor, bounded
by 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32 accumulation.
"""

import numpy as np
import pytest

import oracle as orc
import causal_linear_attention_la_gb300 as la
from causal_linear_attention_la_gb300 import synth
from helpers import STATE_TOL, TOL, Z_TOL, build_lib, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu

PATHS = [la.LA_PATH_AUTO, la.LA_PATH_SIMT]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_lib()
    la.lib()
    yield
    la.la_set_path(la.LA_PATH_AUTO)


def _run(q, k, v, causal, dtype, eps=1e-6, path=la.LA_PATH_AUTO, state=False):
    import torch
    la.la_set_path(path)
    try:
        res = la.forward(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                         causal=causal, eps=eps, return_state=state)
        torch.cuda.synchronize()
    finally:
        la.la_set_path(la.LA_PATH_AUTO)
    return res


@pytest.mark.parametrize("causal", [True, False])
def test_tiny_config_f32(causal):
    # B=1, H=1, N=64, dk=dv=16, fp32, seed 1, eps 1e-6
    q, k, v = synth.qkv(1, 1, 64, 16, 16, seed=1, dtype="f32")
    want = orc.forward_masked(q, k, v, causal=causal, eps=1e-6)
    got = to_host(_run(q, k, v, causal, "f32"))
    err = rel_err(got, want, np.abs(v).max())
    assert err <= TOL["f32"], err


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,N,dk,dv", [
    (1, 1, 1, 16, 16),        # single token
    (1, 2, 31, 32, 16),       # less than one tile, dk != dv
    (2, 1, 129, 64, 64),      # one chunk plus one token
    (1, 1, 1000, 64, 128),    # several segments, ragged tail
    (1, 3, 2000, 128, 128),   # many segments
    (2, 2, 300, 128, 32),
    (1, 1, 4100, 16, 64),
    # tensor-core sizes (bf16, dk = dv in {64, 128}): one token, a
    # partial chunk, exact chunks, many segments with a ragged tail
    (1, 1, 1, 64, 64),
    (1, 2, 127, 128, 128),
    (1, 1, 256, 64, 64),
    (2, 3, 4097, 64, 64),
    (1, 2, 5000, 128, 128),
])
def test_forward_shapes(B, H, N, dk, dv, causal, dtype, path):
    seed = 100 + N + dk + dv
    q, k, v = synth.qkv(B, H, N, dk, dv, seed=seed, dtype=dtype)
    want, S_ref, z_ref = orc.forward_recurrent(q, k, v, causal=causal, eps=1e-6,
                                               return_state=True)
    got, S, z = _run(q, k, v, causal, dtype, path=path, state=True)
    err = rel_err(to_host(got), want, np.abs(v).max())
    assert la.la_device_status(True) == la.LA_OK
    assert err <= TOL[dtype], err
    # final state, relative to its own magnitude (see STATE_TOL)
    s_err = rel_err(to_host(S), S_ref, np.abs(S_ref).max())
    z_err = rel_err(to_host(z), z_ref, np.abs(z_ref).max())
    assert s_err <= STATE_TOL[dtype] and z_err <= Z_TOL[dtype], (s_err, z_err)


def test_forward_eps_zero_and_large():
    q, k, v = synth.qkv(1, 2, 257, 64, 64, seed=9, dtype="bf16")
    for eps in (0.0, 10.0):
        want = orc.forward_recurrent(q, k, v, eps=eps)
        got = to_host(_run(q, k, v, True, "bf16", eps=eps))
        assert rel_err(got, want, np.abs(v).max()) <= TOL["bf16"]


def test_forward_extreme_inputs():
    # large-magnitude q, k: phi saturates to exp(x) ~ 0 or x + 1 ~ large
    rng = np.random.default_rng(3)
    q = (rng.standard_normal((1, 1, 300, 64)) * 8).astype(np.float32)
    k = (rng.standard_normal((1, 1, 300, 64)) * 8).astype(np.float32)
    v = rng.standard_normal((1, 1, 300, 64)).astype(np.float32)
    want = orc.forward_recurrent(q, k, v, eps=1e-6)
    got = to_host(_run(q, k, v, True, "f32"))
    assert rel_err(got, want, np.abs(v).max()) <= TOL["f32"]


def _extreme_bf16(B, H, N, d, seed):
    """bf16 q, k of large magnitude (N(0, 30^2), clipped to +-100: phi runs
    from e^-100 to 101), v of unit scale / 8."""
    rng = np.random.default_rng(seed)
    q = synth.round_to_bf16(np.clip(rng.standard_normal((B, H, N, d)) * 30, -100, 100).astype(np.float32))
    k = synth.round_to_bf16(np.clip(rng.standard_normal((B, H, N, d)) * 30, -100, 100).astype(np.float32))
    v = synth.round_to_bf16((rng.standard_normal((B, H, N, d)) / 8).astype(np.float32))
    return q, k, v


def _hull_ok(out, v, causal):
    """Each output coordinate lies between min(0, min_j v_j) and
    max(0, max_j v_j) over the keys it reads (j <= t causal, all j otherwise):
    the outputs are nonnegative weightings of v with weights summing to at
    most 1 ("Linear Attention: KV를 고정 크기 상태에 누적하기", section
    "점수의 합으로 나누기")."""
    if causal:
        lo = np.minimum(np.minimum.accumulate(v, axis=2), 0.0)
        hi = np.maximum(np.maximum.accumulate(v, axis=2), 0.0)
    else:
        lo = np.minimum(v.min(axis=2, keepdims=True), 0.0)
        hi = np.maximum(v.max(axis=2, keepdims=True), 0.0)
    slack = 2.0 ** -8 * np.abs(v).max()      # the bf16 rounding of the output
    return bool(np.all(out >= lo - slack) and np.all(out <= hi + slack))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_forward_extreme_inputs_tensor_core(d, causal, eps):
    """bf16 inputs of large magnitude through the tensor-core kernels, eps = 0
    included. The kernels' exponential flushes results below the normal range
    to zero; phi is raised to the smallest normal there, so that phi > 0 (the
    feature map's defining property, "Transformers are RNNs" review,
    feature-map table) and every normaliser stays positive. Row 5 of every
    query has all features at -100 (phi(q) = e^-100 in the oracle): the
    output must still be finite and match."""
    import torch
    B, H, N = 1, 2, 700
    q, k, v = _extreme_bf16(B, H, N, d, seed=d + 3 * causal + int(eps > 0))
    q[:, :, 5, :] = -100.0
    want = orc.forward_recurrent(q, k, v, causal=causal, eps=eps)
    got = to_host(_run(q, k, v, causal, "bf16", eps=eps))
    assert la.la_forward_path(d, d, la.LA_BF16, causal) == 1
    assert la.la_device_status(True) == la.LA_OK
    assert np.all(np.isfinite(got))
    assert rel_err(got, want, np.abs(v).max()) <= TOL["bf16"]
    assert _hull_ok(got, v.astype(np.float64), causal)


def test_empty_sequence_zeroes_state():
    import torch
    q = torch.zeros((2, 3, 0, 16), device="cuda")
    v = torch.zeros((2, 3, 0, 32), device="cuda")
    out, S, z = la.forward(q, q, v, return_state=True)
    torch.cuda.synchronize()
    assert out.shape == (2, 3, 0, 32)
    assert float(S.abs().max()) == 0.0 and float(z.abs().max()) == 0.0


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_path_is_taken(d):
    assert la.la_forward_path(d, d, la.LA_BF16, True) == 1
    n0 = la.la_launch_count()
    q, k, v = synth.qkv(1, 1, 300, d, d, seed=77, dtype="bf16")
    want = orc.forward_recurrent(q, k, v)
    got = to_host(_run(q, k, v, True, "bf16"))
    # segment sums (when there is more than one segment), then the chunk loop,
    # which adds up the earlier segments' sums itself
    assert la.la_launch_count() - n0 == 2
    assert la.la_device_status(True) == la.LA_OK
    assert rel_err(got, want, np.abs(v).max()) <= TOL["bf16"]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N", [
    (1, 1, 1),        # one token
    (1, 1, 300),      # one segment, ragged chunk
    (1, 1, 4100),     # many segments, a short last segment
    (6, 10, 2049),    # segments split over several state CTAs, one-token tail
    (2, 3, 9000),
])
def test_noncausal_tensor_core(B, H, N, d):
    """Non-causal: every query reads the whole-sequence state S_N, z_N; the
    state pass sums all segments and a second kernel applies the total."""
    assert la.la_forward_path(d, d, la.LA_BF16, False) == 1
    q, k, v = synth.qkv(B, H, N, d, d, seed=500 + N + d, dtype="bf16")
    want, S_ref, z_ref = orc.forward_recurrent(q, k, v, causal=False, eps=1e-6,
                                               return_state=True)
    n0 = la.la_launch_count()
    got, S, z = _run(q, k, v, False, "bf16", state=True)
    assert la.la_launch_count() - n0 == 2
    assert la.la_device_status(True) == la.LA_OK
    err = rel_err(to_host(got), want, np.abs(v).max())
    assert err <= TOL["bf16"], err
    s_err = rel_err(to_host(S), S_ref, np.abs(S_ref).max())
    z_err = rel_err(to_host(z), z_ref, np.abs(z_ref).max())
    assert s_err <= STATE_TOL["bf16"] and z_err <= Z_TOL["bf16"], (s_err, z_err)


def test_state_pass_split_over_ctas():
    """60 sequences of 2048 tokens: two segments per sequence, and the segment
    sums of the first are split over two CTAs of the state pass (its workspace
    then holds more records than the CUDA-core plan). Sampled heads, final
    state included, are checked against the oracle."""
    import torch
    B, H, N, d = 6, 10, 2048, 64
    ws_tc = la.la_forward_workspace_size(B, H, N, d, d, 1, la.LA_BF16)
    ws_f32 = la.la_forward_workspace_size(B, H, N, d, d, 1, la.LA_F32)
    assert ws_tc > ws_f32
    q, k, v = synth.qkv(B, H, N, d, d, seed=606, dtype="bf16")
    out, S, z = _run(q, k, v, True, "bf16", state=True)
    assert la.la_device_status(True) == la.LA_OK
    out, S, z = to_host(out), to_host(S), to_host(z)
    for b, h in [(0, 0), (2, 5), (5, 9)]:
        want, S_w, z_w = orc.forward_recurrent(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                               v[b:b + 1, h:h + 1], return_state=True)
        assert rel_err(out[b:b + 1, h:h + 1], want, np.abs(v).max()) <= TOL["bf16"]
        assert rel_err(S[b, h], S_w[0, 0], np.abs(S_w).max()) <= STATE_TOL["bf16"]
        assert rel_err(z[b, h], z_w[0, 0], np.abs(z_w).max()) <= Z_TOL["bf16"]


# Balanced pieces (causal, d = 128, bf16, no final state): the heads' chunks
# laid end to end and cut into equal pieces, one CTA each. Shapes: pieces of
# two chunks over heads of 5 and 7 chunks with ragged last chunks (most
# pieces end one head and start the next), heads of 33 chunks (pieces of 5,
# up to 7 records summed per piece), and the
# bench's B=2 H=16 N=8192 split (14-chunk pieces, piece 32 starting exactly
# at head 7, a short last piece).
@pytest.mark.parametrize("B,H,N,heads", [
    (3, 17, 544, None),
    (1, 39, 803, None),
    (1, 22, 4224, None),
    (2, 16, 8192, [0, 6, 7, 8, 15, 16, 31]),
])
def test_forward_balanced_pieces(B, H, N, heads):
    import torch
    d = 128
    plan = la.forward_plan(B, H, N, d, d)
    assert plan["pieces"] > 0, plan
    assert la.forward_plan(B, H, N, d, d, final_state=True)["pieces"] == 0
    q, k, v = synth.qkv(B, H, N, d, d, seed=840 + N, dtype="bf16")
    n0 = la.la_launch_count()
    got = to_host(_run(q, k, v, True, "bf16"))
    assert la.la_launch_count() - n0 == 2
    assert la.la_device_status(True) == la.LA_OK
    flat = lambda x: x.reshape(B * H, N, -1)
    sel = list(range(B * H)) if heads is None else heads
    want = orc.forward_recurrent(flat(q)[None, sel], flat(k)[None, sel], flat(v)[None, sel], eps=1e-6)
    err = rel_err(flat(got)[sel], want[0], np.abs(v).max())
    assert err <= TOL["bf16"], err
    # with a final state the same call runs by segments: same outputs
    got2, S, z = _run(q, k, v, True, "bf16", state=True)
    err2 = rel_err(flat(to_host(got2))[sel], want[0], np.abs(v).max())
    assert err2 <= TOL["bf16"], err2
