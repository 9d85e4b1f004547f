"""The bounded waits of the tensor-core kernels, on the GPU, without a fault.

la_test_timeout_next_forward makes the MMA-issuing thread of the next causal
tensor-core forward wait on an mbarrier that nothing ever completes. Its wait
must give up after the kernels' limit (2 s), the whole CTA must wind down
(every other warp sees the abort flag in its own bounded waits, in-flight
copies are drained, tensor memory is freed), and the per-device status word
must read LA_ERR_TIMEOUT. The context stays usable: the next call runs
normally and matches the oracle.
"""

import time

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


@pytest.mark.parametrize("d", [64, 128])
def test_bounded_wait_gives_up_and_the_next_call_runs(d):
    import torch
    q, k, v = synth.qkv(1, 1, 300, d, d, seed=55 + d, dtype="bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    la.forward(qd, kd, vd)            # warm: build, tensor maps, attributes
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    la.la_test_timeout_next_forward()
    t0 = time.perf_counter()
    la.forward(qd, kd, vd)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert la.la_device_status(True) == la.LA_ERR_TIMEOUT
    assert 1.5 < waited < 30.0, waited
    # the switch was one-shot and the context is intact
    got = la.forward(qd, kd, vd)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    want = orc.forward_recurrent(q, k, v, eps=1e-6)
    assert rel_err(to_host(got), want, np.abs(v).max()) <= TOL["bf16"]
