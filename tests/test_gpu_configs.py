"""Parity at the full benchmark sizes, in the launch configuration the bench
times (default path, one call per pass):

* causal forward B=4 H=8 N=4096 d=64 bf16: every output vs the oracle recurrence
* causal forward B=2 H=16 N=32768 d=128 bf16, as the bench runs it
  (balanced pieces) and with the final state (segments): three whole heads
  (every one of their 32768 outputs, and the final state) against the
  oracle recurrence, plus outputs sampled at every piece's first and last
  chunk and at random, each computed one by one by the oracle's definition
* decode: fp32 states from a bf16 prefill of N=131072 tokens on B=1 H=16,
  replicated to B=64 x H=32, then 1024 one-token steps; every state's output
  for the first 8 steps, and 64 sampled states' outputs for all 1024 steps
  (and their final states)
* forward + backward B=4 H=8 N=8192 d=64 bf16: every gradient vs the oracle,
  causal and non-causal, with the backward recomputing the state records and
  reusing the forward's (la_backward_saved, as the bench runs it)
* decay-gated forward B=4 H=8 N=4096 d=64 bf16 (per-head factors 0.9 ..
  0.999, as the bench): every output and the final state vs the oracle's
  decayed recurrence
* forward through the host-buffer call at B=4 H=8 N=4096 d=64 (the bench's
  end-to-end line, two sequence groups): every output vs the oracle
"""

import numpy as np
import pytest

import oracle as orc
import causal_linear_attention_la_gb300 as la
from causal_linear_attention_la_gb300 import synth
from helpers import STATE_TOL, TOL, Z_TOL, Z_TOL_DECAY_BF16, build_lib, grad_errors, grad_tol, grads_ok, rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_lib()
    la.lib()


def test_forward_b4_h8_n4096_d64():
    import torch
    q, k, v = synth.qkv(4, 8, 4096, 64, 64, seed=2, dtype="bf16")
    want = orc.forward_recurrent(q, k, v, eps=1e-6)
    got = la.forward(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"))
    torch.cuda.synchronize()
    err = rel_err(to_host(got), want, np.abs(v).max())
    assert err <= TOL["bf16"], err


def test_forward_b2_h16_n32768_d128():
    import torch
    B, H, N, d = 2, 16, 32768, 128
    q, k, v = synth.qkv(B, H, N, d, d, seed=3, dtype="bf16")
    qd, kd, vd = to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16")
    # as the bench runs it (no final state): 152 balanced pieces of 54 chunks
    plan = la.forward_plan(B, H, N, d, d)
    assert (plan["pieces"], plan["piece_len"]) == (152, 54), plan
    out_p = la.forward(qd, kd, vd).float().cpu().numpy()
    # with the final state: by segments
    out, S, z = la.forward(qd, kd, vd, return_state=True)
    torch.cuda.synchronize()
    out = out.float().cpu().numpy()
    vmax = np.abs(v).max()
    # three whole heads, every output of both calls and the final state,
    # element by element (head (0, 7) holds piece boundaries at chunks 10,
    # 64, 118, 172 and 226 of its 256)
    for b, h in ((0, 0), (0, 7), (1, H - 1)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        want, S_w, z_w = orc.forward_recurrent(q[sl], k[sl], v[sl], eps=1e-6, return_state=True)
        assert rel_err(out_p[sl], want, vmax) <= TOL["bf16"], (b, h)
        assert rel_err(out[sl], want, vmax) <= TOL["bf16"], (b, h)
        assert rel_err(to_host(S[b, h]), S_w[0, 0], np.abs(S_w).max()) <= STATE_TOL["bf16"]
        assert rel_err(to_host(z[b, h]), z_w[0, 0], np.abs(z_w).max()) <= Z_TOL["bf16"]
    rng = np.random.default_rng(0)
    worst = 0.0
    picks = [(b, h, t) for b in range(B) for h in (0, H - 1) for t in (0, 127, 128, N - 1)]
    # the first and last token of every piece
    for i in range(plan["pieces"]):
        for g in (i * 54, min(B * H * 256, i * 54 + 54) - 1):
            bh, c = divmod(g, 256)
            picks += [(bh // H, bh % H, 128 * c), (bh // H, bh % H, 128 * c + 127)]
    picks += [(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N)))
              for _ in range(48)]
    for b, h, t in picks:
        want = orc.output_at(q[b, h], k[b, h], v[b, h], t, eps=1e-6)
        worst = max(worst, rel_err(out[b, h, t], want, vmax), rel_err(out_p[b, h, t], want, vmax))
    assert worst <= TOL["bf16"], worst
    for b, h in ((0, 0), (1, H - 1)):
        fk = orc.phi_elu1(k[b, h])
        S_ref = fk.T @ v[b, h].astype(np.float64)
        assert rel_err(to_host(S[b, h]), S_ref, np.abs(S_ref).max()) <= STATE_TOL["bf16"]
        assert rel_err(to_host(z[b, h]), fk.sum(0), fk.sum(0).max()) <= Z_TOL["bf16"]


def test_decode_b64_h32_d128_from_prefill_n131072():
    import torch
    d, Hp, Np = 128, 16, 131072
    B, H = 64, 32
    steps, full_steps = 1024, 8
    qp, kp, vp = synth.qkv(1, Hp, Np, d, d, seed=4, dtype="bf16")
    _, Sp, zp = la.forward(to_dev(qp, "bf16"), to_dev(kp, "bf16"), to_dev(vp, "bf16"),
                           return_state=True)
    torch.cuda.synchronize()
    # oracle prefill states of every prefill head, fp64
    S_or = np.stack([orc.phi_elu1(kp[0, h]).T @ vp[0, h].astype(np.float64) for h in range(Hp)])
    z_or = np.stack([orc.phi_elu1(kp[0, h]).sum(0) for h in range(Hp)])
    del qp, kp, vp
    assert rel_err(to_host(Sp[0]), S_or, np.abs(S_or).max()) <= STATE_TOL["bf16"]
    assert rel_err(to_host(zp[0]), z_or, np.abs(z_or).max()) <= Z_TOL["bf16"]
    # state (b, h) starts from prefill head (b*H + h) mod Hp
    src = (np.arange(B * H) % Hp)
    S = Sp[0][torch.from_numpy(src).cuda()].reshape(B, H, d, d).contiguous()
    z = zp[0][torch.from_numpy(src).cuda()].reshape(B, H, d).contiguous()
    S_ref = S_or[src].reshape(B, H, d, d)
    z_ref = z_or[src].reshape(B, H, d)
    # 64 sampled states followed through all steps
    pick = np.sort(np.random.default_rng(7).choice(B * H, 64, replace=False))
    idx = (pick // H, pick % H)
    S_s, z_s = S_ref[idx].copy(), z_ref[idx].copy()
    worst_all = worst_s = 0.0
    for step in range(steps):
        q, k, v = synth.decode_token(B, H, d, d, seed=1000, step=step)
        out = la.decode_step(S, z, to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"))
        torch.cuda.synchronize()
        got = to_host(out)
        vmax = np.abs(v).max()
        if step < full_steps:   # every state
            S_ref, z_ref, o_ref = orc.decode_step(S_ref, z_ref, q, k, v)
            worst_all = max(worst_all, rel_err(got, o_ref, vmax))
        S_s, z_s, o_s = orc.decode_step(S_s, z_s, q[idx], k[idx], v[idx])
        worst_s = max(worst_s, rel_err(got[idx], o_s, vmax))
    assert worst_all <= TOL["bf16"], worst_all
    assert worst_s <= TOL["bf16"], worst_s
    # the sampled states after all steps (fp32 in-place updates)
    S_h = to_host(S)[idx]
    z_h = to_host(z)[idx]
    assert rel_err(S_h, S_s, np.abs(S_s).max()) <= STATE_TOL["bf16"]
    assert rel_err(z_h, z_s, np.abs(z_s).max()) <= Z_TOL["bf16"]


def test_forward_backward_b4_h8_n8192_d64():
    import torch
    B, H, N, d = 4, 8, 8192, 64
    q, k, v = synth.qkv(B, H, N, d, d, seed=5, dtype="bf16")
    g = synth.upstream_grad(B, H, N, d, seed=5, dtype="bf16")
    qd, kd, vd, gd = (to_dev(x, "bf16") for x in (q, k, v, g))
    out = la.forward(qd, kd, vd)
    grads = la.backward(qd, kd, vd, gd)
    # as the bench runs it: the backward reusing the forward's state records
    ws = torch.empty(la.la_forward_workspace_size(B, H, N, d, d, 1, la.LA_BF16), dtype=torch.uint8, device="cuda")
    la.forward(qd, kd, vd, workspace=ws)
    grads_saved = la.backward_saved(qd, kd, vd, gd, ws)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    want_o = orc.forward_recurrent(q, k, v, eps=1e-6)
    assert rel_err(to_host(out), want_o, np.abs(v).max()) <= TOL["bf16"]
    want = orc.backward_recurrent(q, k, v, g, eps=1e-6)
    errs = grad_errors(grads, want)
    assert grads_ok(errs, grad_tol("bf16", True)), errs
    errs = grad_errors(grads_saved, want)
    assert grads_ok(errs, grad_tol("bf16", True)), errs


def test_forward_backward_noncausal_b4_h8_n8192_d64():
    import torch
    B, H, N, d = 4, 8, 8192, 64
    q, k, v = synth.qkv(B, H, N, d, d, seed=5, dtype="bf16")
    g = synth.upstream_grad(B, H, N, d, seed=5, dtype="bf16")
    qd, kd, vd, gd = (to_dev(x, "bf16") for x in (q, k, v, g))
    out = la.forward(qd, kd, vd, causal=False)
    grads = la.backward(qd, kd, vd, gd, causal=False)
    ws = torch.empty(la.la_forward_workspace_size(B, H, N, d, d, 0, la.LA_BF16), dtype=torch.uint8, device="cuda")
    la.forward(qd, kd, vd, causal=False, workspace=ws)
    grads_saved = la.backward_saved(qd, kd, vd, gd, ws, causal=False)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    want_o = orc.forward_recurrent(q, k, v, causal=False, eps=1e-6)
    assert rel_err(to_host(out), want_o, np.abs(v).max()) <= TOL["bf16"]
    want = orc.backward_recurrent(q, k, v, g, causal=False, eps=1e-6)
    errs = grad_errors(grads, want)
    assert grads_ok(errs, grad_tol("bf16", True)), errs
    errs = grad_errors(grads_saved, want)
    assert grads_ok(errs, grad_tol("bf16", True)), errs


def test_forward_decay_b4_h8_n4096_d64():
    import torch
    B, H, N, d = 4, 8, 4096, 64
    q, k, v = synth.qkv(B, H, N, d, d, seed=2, dtype="bf16")
    alpha = np.linspace(0.9, 0.999, H).astype(np.float32)
    out, S, z = la.forward_decay(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"),
                                 torch.from_numpy(alpha).cuda(), return_state=True)
    torch.cuda.synchronize()
    assert la.la_device_status(True) == la.LA_OK
    S_w, z_w, o_w = orc.decode_steps_decay(np.zeros((B, H, d, d)), np.zeros((B, H, d)), q, k, v,
                                           alpha=alpha.astype(np.float64)[None, :])
    assert rel_err(to_host(out), o_w, np.abs(v).max()) <= TOL["bf16"]
    assert rel_err(to_host(S), S_w, np.abs(S_w).max()) <= STATE_TOL["bf16"]
    assert rel_err(to_host(z), z_w, np.abs(z_w).max()) <= Z_TOL_DECAY_BF16


def test_forward_host_b4_h8_n4096_d64():
    import torch
    q, k, v = synth.qkv(4, 8, 4096, 64, 64, seed=2, dtype="bf16")
    hq, hk, hv = (to_dev(x, "bf16").cpu().pin_memory() for x in (q, k, v))
    got = la.forward_host(hq, hk, hv, slices=2)
    torch.cuda.synchronize()
    want = orc.forward_recurrent(q, k, v, eps=1e-6)
    assert rel_err(to_host(got), want, np.abs(v).max()) <= TOL["bf16"]
