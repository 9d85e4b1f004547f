"""la_forward_host (host buffers, pipelined copies) vs the oracle and vs
la_forward on each slice of sequences."""

import numpy as np
import pytest

import oracle as orc
import causal_linear_attention_la_gb300 as la
from causal_linear_attention_la_gb300 import synth
from helpers import TOL, build_lib, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_lib()
    la.lib()
    yield


def _host(x, dtype, pin=True):
    import torch
    t = to_dev(x, dtype).cpu()
    return t.pin_memory() if pin else t


@pytest.mark.parametrize("dtype,d,causal", [("bf16", 64, True), ("bf16", 64, False),
                                            ("bf16", 128, True), ("f32", 32, True)])
@pytest.mark.parametrize("B,H,N,slices", [(2, 3, 700, 4), (1, 1, 129, 3), (4, 8, 1024, 4), (1, 5, 300, 2)])
def test_forward_host_matches_oracle_and_slices(B, H, N, slices, dtype, d, causal):
    import torch
    q, k, v = synth.qkv(B, H, N, d, d, seed=N + 7 * H + d, dtype=dtype)
    hq, hk, hv = (_host(x, dtype) for x in (q, k, v))
    out = la.forward_host(hq, hk, hv, causal=causal, slices=slices)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    want = orc.forward_recurrent(q, k, v, causal=causal)
    assert rel_err(to_host(out), want, np.abs(v).max()) <= TOL[dtype]
    # each slice is la_forward over its own sequences: the same bits
    BH = B * H
    S = min(slices, BH)
    base, extra = divmod(BH, S)
    flat = [x.reshape(BH, N, d) for x in (hq, hk, hv)]
    got = out.reshape(BH, N, d)
    s0 = 0
    for i in range(S):
        cnt = base + (1 if i < extra else 0)
        sl = [x[s0:s0 + cnt].reshape(1, cnt, N, d).cuda() for x in flat]
        ref = la.forward(*sl, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(ref.cpu().reshape(cnt, N, d), got[s0:s0 + cnt]), i
        s0 += cnt


def test_forward_host_pageable_and_side_stream():
    """Pageable host memory works (copies then block the caller); the call
    is ordered on the given stream and its output is complete when the
    stream reaches the point after it."""
    import torch
    B, H, N, d = 2, 4, 513, 64
    q, k, v = synth.qkv(B, H, N, d, d, seed=99, dtype="bf16")
    hq, hk, hv = (_host(x, "bf16", pin=False) for x in (q, k, v))
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        la.forward_host(hq, hk, hv, out=out, slices=3)
    side.synchronize()
    want = orc.forward_recurrent(q, k, v)
    assert rel_err(out.float().numpy(), want, np.abs(v).max()) <= TOL["bf16"]
    # repeated calls on one workspace and pinned buffers give the same bits
    pq, pk, pv = (x.pin_memory() for x in (hq, hk, hv))
    ws = torch.empty(la.la_forward_host_workspace_size(B, H, N, d, d, 1, la.LA_BF16, 2),
                     dtype=torch.uint8, device="cuda")
    o1 = la.forward_host(pq, pk, pv, slices=2, workspace=ws)
    o2 = la.forward_host(pq, pk, pv, slices=2, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
