"""la_forward_noalloc, the forward entry point for callers that cannot
allocate device memory (operator hosts that own all device memory and hand an
operator only its inputs and outputs, latency-critical loops that cannot
afford cudaMalloc's implicit synchronisation): its scratch is a static device
array inside the library instead of a caller-provided workspace.

Through the C ABI, calls in a row must each match la_forward (with a
caller-allocated workspace) on the same inputs: within the parity tolerance
of the other tests, and in fact bit for bit, since both run the same kernels
on the same inputs. Between two calls of one shape come calls that change the
shape, the causality and the dtype, so that every call must rewrite each
record it reads whatever the previous call left in the shared array. A
problem whose scratch exceeds the static array must be rejected before
anything is launched. Collected last so that a failure here never hides the
results of the other GPU tests.
"""

import numpy as np
import pytest

import causal_linear_attention_la_gb300 as la
from causal_linear_attention_la_gb300 import synth
from helpers import STATE_TOL, TOL, Z_TOL, build_lib, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_lib()
    la.lib()


def _noalloc(q, k, v, causal, code, state=True):
    import torch
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    out = torch.empty((B, H, N, dv), dtype=q.dtype, device=q.device)
    S = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if state else None
    z = torch.empty((B, H, dk), dtype=torch.float32, device=q.device) if state else None
    st = la.la_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               B, H, N, dk, dv, causal, 1e-6, code,
                               S.data_ptr() if state else None, z.data_ptr() if state else None,
                               torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, la.lib().la_last_error()
    return out, S, z


# (dtype, (B, H, N, dk, dv), causal, seed, final state): the first shape
# twice, with a different shape, a non-causal call, the CUDA-core (fp32) path
# and a d = 128 call without a final state (balanced pieces: the records are
# laid out per piece) between
CALLS = [
    ("bf16", (4, 8, 4096, 64, 64), True, 41, True),
    ("bf16", (2, 3, 1000, 64, 64), False, 43, True),
    ("f32", (1, 2, 1000, 32, 64), True, 44, True),
    ("bf16", (3, 17, 640, 128, 128), True, 46, False),
    ("bf16", (1, 2, 5000, 128, 128), True, 45, True),
    ("bf16", (4, 8, 4096, 64, 64), True, 42, True),
]


def test_noalloc_matches_forward_on_calls_in_a_row():
    import torch
    for dtype, (B, H, N, dk, dv), causal, seed, state in CALLS:
        code = la.LA_BF16 if dtype == "bf16" else la.LA_F32
        assert la.la_forward_workspace_size(B, H, N, dk, dv, causal, code) <= la.LA_NOALLOC_SCRATCH_BYTES
        q, k, v = synth.qkv(B, H, N, dk, dv, seed=seed, dtype=dtype)
        qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
        if not state:
            assert la.forward_plan(B, H, N, dk, dv, causal=causal, dtype=code)["pieces"] > 0
            ref = la.forward(qd, kd, vd, causal=causal)
            out, _, _ = _noalloc(qd, kd, vd, causal, code, state=False)
            torch.cuda.synchronize()
            assert la.la_device_status(True) == la.LA_OK
            assert rel_err(to_host(out), to_host(ref), np.abs(v).max()) <= TOL[dtype]
            assert torch.equal(out, ref), (dtype, B, H, N, causal)
            continue
        ref, S_ref, z_ref = la.forward(qd, kd, vd, causal=causal, return_state=True)
        out, S, z = _noalloc(qd, kd, vd, causal, code)
        torch.cuda.synchronize()
        assert la.la_device_status(True) == la.LA_OK
        ref_h, S_ref_h, z_ref_h = to_host(ref), to_host(S_ref), to_host(z_ref)
        assert rel_err(to_host(out), ref_h, np.abs(v).max()) <= TOL[dtype]
        assert rel_err(to_host(S), S_ref_h, np.abs(S_ref_h).max()) <= STATE_TOL[dtype]
        assert rel_err(to_host(z), z_ref_h, np.abs(z_ref_h).max()) <= Z_TOL[dtype]
        assert torch.equal(out, ref), (dtype, B, H, N, causal)
        assert torch.equal(S, S_ref) and torch.equal(z, z_ref), (dtype, B, H, N, causal)


def test_noalloc_rejects_oversized_problem():
    B, H, N, d = 2, 16, 32768, 128
    need = la.la_forward_workspace_size(B, H, N, d, d, 1, la.LA_BF16)
    assert need > la.LA_NOALLOC_SCRATCH_BYTES
    st = la.la_forward_noalloc(None, None, None, None, B, H, N, d, d, 1, 1e-6,
                               la.LA_BF16, None, None, None)
    assert st == la.LA_ERR_INVALID_ARG
    assert b"static array" in la.lib().la_last_error()
