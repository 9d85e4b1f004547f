#!/usr/bin/env python3
"""Benchmark of the GB300 causal linear-attention library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0). The headline workload is the largest
single-GPU forward: causal, B=2 H=16 N=32768 dk=dv=128 bf16 (one step = one
la_forward over the batch: the per-segment state sums and the chunked output
kernel, which adds up the earlier segments' records). `value` is tokens/s (a
token = one position of one sequence, all heads) with inputs resident in HBM;
`e2e` is the same metric through the host-buffer C-ABI call la_forward_host
(pinned host q, k, v, out; every step's host<->device copies inside the timed
region; sequence groups overlap their copies with their neighbours' compute,
and the unpipelined call is reported beside it). The other workloads of the
method are measured in the same run and reported under "sections": the
causal forward B=4 H=8 N=4096 d=64, the decode step on B=64 x H=32 fp32
states of d=128 (1024 steps in a CUDA graph), the same decode with 16 tokens
per call (64 calls of la_decode_steps), the decay-gated and delta-rule
variants in the same shape, forward + backward B=4 H=8 N=8192 d=64 (causal
and not; the backward reuses the forward's state records through
la_backward_saved), the decay-gated forward in the B=4 H=8 N=4096 d=64
shape, and the chunked delta rule over B=2 H=16 N=8192 d=128 (CUDA cores,
against the fp32 FMA rate at the sampled SM clock).

Timing: W eager warm-up steps, then the K timed steps are captured once in a
CUDA graph and replayed, bracketed by CUDA events on the launching stream
(and a barrier + synchronize on both sides under torchrun). Inputs rotate
over enough copies that each step reads data not left in the 129 MB L2.
Kernel spans (for the roofline) come from events the library records around
its kernels (la_profile_enable), in a second graph of the same K steps.

cpu_baseline and --impl reference time the fp64 CPU oracle on a bounded
sample of the same workload (a prefix of every sequence), its sequences
spread over a process pool on all host cores: the reference implementation
of this method.

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path has no cross-GPU exchange); value = all ranks' tokens / max rank time.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal linear-attn tokens/s & TFLOP/s (fwd, bwd) + decode GB/s vs GB300 roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOADS = {
    "fwd_b4_h8_n4096_d64": dict(kind="forward", B=4, H=8, N=4096, dk=64, dv=64, causal=True, seed=2),
    "fwd_b2_h16_n32768_d128": dict(kind="forward", B=2, H=16, N=32768, dk=128, dv=128, causal=True, seed=3),
    "decode_b64_h32_d128": dict(kind="decode", B=64, H=32, dk=128, dv=128, seed=4,
                                prefill=dict(B=1, H=16, N=131072), steps=1024),
    "fwdbwd_b4_h8_n8192_d64": dict(kind="fwdbwd", B=4, H=8, N=8192, dk=64, dv=64, causal=True, seed=5),
    # the same shape without the causal mask (every query reads the whole sequence)
    "fwdbwd_nc_b4_h8_n8192_d64": dict(kind="fwdbwd", B=4, H=8, N=8192, dk=64, dv=64, causal=False, seed=5),
    # decay-gated forward (per-head factors 0.9 .. 0.999), the headline shape
    "fwd_decay_b4_h8_n4096_d64": dict(kind="forward", B=4, H=8, N=4096, dk=64, dv=64, causal=True, seed=2,
                                      decay=True),
    # the same states, 16 tokens per call (la_decode_steps): 64 calls = 1024 tokens
    "decode16_b64_h32_d128": dict(kind="decode", B=64, H=32, dk=128, dv=128, seed=4,
                                  prefill=dict(B=1, H=16, N=131072), steps=64, tokens=16),
    # the state-update variants on the same states, 16 tokens per call
    "decay16_b64_h32_d128": dict(kind="decode", B=64, H=32, dk=128, dv=128, seed=4,
                                 prefill=dict(B=1, H=16, N=131072), steps=64, tokens=16,
                                 variant="decay"),
    # the delta rule over whole sequences, chunk by chunk (la_forward_delta)
    "deltafwd_b2_h16_n8192_d128": dict(kind="delta_fwd", B=2, H=16, N=8192, dk=128, dv=128, seed=6),
    # 256 heads: the tensor-core group kernel
    "deltafwd_b8_h32_n2048_d128": dict(kind="delta_fwd", B=8, H=32, N=2048, dk=128, dv=128, seed=6),
    "delta16_b64_h32_d128": dict(kind="decode", B=64, H=32, dk=128, dv=128, seed=4,
                                 prefill=dict(B=1, H=16, N=131072), steps=64, tokens=16,
                                 variant="delta"),
}
MAIN = "fwd_b2_h16_n32768_d128"
EPS = 1e-6
E2E_SLICES = 8          # la_forward_host: sequence groups whose copies overlap compute (best measured on the headline shape)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_helpers(world, device):
    """barrier() and max_over_ranks(x) over the initialised process group of
    `world` ranks (plain functions for one rank). `device`: where the
    all-reduce tensor lives ("cuda" under NCCL, "cpu" under gloo)."""
    if world <= 1:
        return (lambda: None), (lambda x: x)
    import torch
    import torch.distributed as dist

    def barrier():
        dist.barrier()

    def max_over_ranks(x):
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_over_ranks


def job_throughput(world, units_per_rank, seconds):
    """Whole-job throughput: the units every rank processed (each rank does
    the same work: weak scaling) over the slowest rank's time."""
    return world * units_per_rank / seconds


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        rows = [r for r in self.samples if num(r[1]) is not None]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(num(r[1]) for r in loaded),
                "sm_max_mhz": max(num(r[2]) or 0 for r in rows),
                "reasons": reasons, "samples": len(loaded)}


# source files of the kernels behind each measured span (the traffic lines in
# profiles/ncu_dram_traffic.txt carry the digest of these files)
_COMMON_TC = ["la_tc_common.cuh", "la_sm100.cuh", "la_internal.cuh"]
KERNEL_SOURCES = {
    "fwd_output": ["la_tc_fwd.cu"] + _COMMON_TC,
    "bwd": ["la_tc_bwd.cu"] + _COMMON_TC,
    "decode": ["la_decode.cu", "la_internal.cuh"],
    "decodetc": ["la_decode_tc.cu", "la_variants.cuh"] + _COMMON_TC,
    "variants": ["la_variants.cu", "la_variants.cuh", "la_internal.cuh"],
}


def ncu_traffic(span):
    """DRAM bytes per launch of a kernel span from the committed ncu summary,
    if it was taken on the kernel sources currently built (digest match), else None."""
    from causal_linear_attention_la_gb300.build import kernel_digest
    path = os.path.join(ROOT, "profiles", "ncu_dram_traffic.txt")
    key = next((k for k in KERNEL_SOURCES if span.startswith(k + "_")), None)
    if key is None:
        return None
    try:
        digest = kernel_digest(KERNEL_SOURCES[key])
        for line in open(path):
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == span and parts[1] == digest[:16]:
                return float(parts[3])
    except OSError:
        pass
    return None


# ---------------------------------------------------------------------------
# algorithmic work models (per launch / per step)
# ---------------------------------------------------------------------------


def fwd_bytes(w, elt=2):
    """Minimum HBM bytes of one forward: read q, k, v once, write out once."""
    return w["B"] * w["H"] * w["N"] * (2 * w["dk"] + 2 * w["dv"]) * elt


def fwd_flops(w):
    """Algorithmic flops of the recurrence: update + read, 2 * 2 * dk * dv per token-head."""
    return 4.0 * w["dk"] * w["dv"] * w["B"] * w["H"] * w["N"]


def fwd_mma_flops(w, C=128):
    """Flops the tensor cores execute in the causal chunk loop, per launch:
    per 128-token chunk and head, d = 64: [P | O | dz] (M128 N208 K64),
    [S^T ; z] += [V^T ; 1] phi(K) (M128 N64 K128), [O | den] += P [V | 1]
    (M128 N80 K128); d = 128: P, O, the state update and P V, each M128
    N128 K128."""
    chunks = w["B"] * w["H"] * -(-w["N"] // C)
    if w["dk"] == 64:
        per = 2 * 128 * (208 * 64 + 64 * 128 + 80 * 128)
    else:
        per = 4 * 2 * 128 * 128 * w["dk"]
    return float(chunks * per)


def tensor_line(w, span_ms, peaks):
    """Tensor-pipe use of the chunk loop: executed MMA flops / its live span,
    against the measured bf16 dense peak (burst: the kernel is timed alone)."""
    ach = fwd_mma_flops(w) / (span_ms / 1e3) / 1e12
    return {"achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"], "kernel": "fwd_output",
            "flops_per_launch": fwd_mma_flops(w),
            "flops": "MMA flops executed by the chunk loop (not the recurrence's 4 dk dv per token-head)"}


def bwd_bytes(w, elt=2):
    """Minimum HBM bytes of one backward: read q, k, v, dout; write dq, dk, dv."""
    return w["B"] * w["H"] * w["N"] * (4 * w["dk"] + 3 * w["dv"]) * elt


def decode_state_bytes(w):
    """S and z read and written once per step (call), fp32; the delta rule keeps no z."""
    zwords = 0 if w.get("variant") == "delta" else w["dk"]
    return w["B"] * w["H"] * (w["dk"] * w["dv"] + zwords) * 4 * 2


def delta_flops(w):
    """Algorithmic flops of the delta rule token by token: the read with the
    key, the rank-one write and the read with the query, 3 * 2 * dk * dv per
    token-head."""
    return 6.0 * w["dk"] * w["dv"] * w["B"] * w["H"] * w["N"]


def fp32_peak_tflops(sm_mhz):
    """CUDA-core fp32 rate: 152 SMs x 128 FMA lanes x 2 flops at the SM clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def decode_io_bytes(w, elt=2):
    return w["B"] * w["H"] * (2 * w["dk"] + 2 * w["dv"]) * elt


# ---------------------------------------------------------------------------
# GPU timing
# ---------------------------------------------------------------------------


def _graph_time(step_fn, K, stream, barrier, profile=False):
    """Capture K steps in a CUDA graph, replay once untimed, then time one replay."""
    import torch
    import causal_linear_attention_la_gb300 as la
    g = torch.cuda.CUDAGraph()
    if profile:
        la.la_profile_enable(1)   # the captured launches carry event-record nodes
    n0 = la.la_launch_count()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for i in range(K):
            step_fn(i)
    launches = la.la_launch_count() - n0
    if profile:
        la.la_profile_enable(0)   # keep the captured spans, record no new ones
    g.replay()
    torch.cuda.synchronize()
    if profile:
        g.replay()                # the events now hold this replay's times
        torch.cuda.synchronize()
        return None, launches, la.la_profile_read()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1), launches, None


def _span_stats(spans):
    out = {}
    for name, ms in spans:
        if ms >= 0:
            out.setdefault(name, []).append(ms)
    return {k: {"launches": len(v), "avg_ms": float(np.mean(v)), "total_ms": float(np.sum(v))}
            for k, v in out.items()}


def _rotations(bytes_per_set):
    return max(1, int(np.ceil(2 * L2_BYTES / max(bytes_per_set, 1))))


def run_forward(w, K, W, barrier, with_bwd=False):
    import torch
    import causal_linear_attention_la_gb300 as la
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(w["seed"])
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    per_set = fwd_bytes(w) + (bwd_bytes(w) if with_bwd else 0)
    R = _rotations(per_set)

    def rnd(shape, scale):
        return (torch.randn(shape, generator=gen, device=dev) * scale).to(torch.bfloat16)

    sets = []
    for _ in range(R):
        s = dict(q=rnd((B, H, N, dk), dk ** -0.5), k=rnd((B, H, N, dk), dk ** -0.5),
                 v=rnd((B, H, N, dv), dv ** -0.5),
                 out=torch.empty((B, H, N, dv), dtype=torch.bfloat16, device=dev))
        if with_bwd:
            s["g"] = rnd((B, H, N, dv), 1.0)
            s["dq"] = torch.empty_like(s["q"])
            s["dk"] = torch.empty_like(s["k"])
            s["dv"] = torch.empty_like(s["v"])
        sets.append(s)
    code = la.LA_BF16
    ws_f = la.la_forward_workspace_size(B, H, N, dk, dv, w["causal"], code)
    ws_b = la.la_backward_workspace_size(B, H, N, dk, dv, w["causal"], code) if with_bwd else 0
    ws = torch.empty(max(ws_f, 1), dtype=torch.uint8, device=dev)
    # the backward keeps its own scratch and reads the forward's state
    # records from `ws` (la_backward_saved: save-for-backward)
    wsb = torch.empty(max(ws_b, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    alpha = torch.linspace(0.9, 0.999, H, device=dev)       # decay: per-head factors

    def step(i):
        s = sets[i % R]
        sp = torch.cuda.current_stream().cuda_stream
        if w.get("decay"):
            st = la.la_forward_decay(s["q"].data_ptr(), s["k"].data_ptr(), s["v"].data_ptr(),
                                     s["out"].data_ptr(), B, H, N, dk, dv, alpha.data_ptr(), EPS, code,
                                     None, None, ws.data_ptr(), ws.numel(), sp)
        else:
            st = la.la_forward(s["q"].data_ptr(), s["k"].data_ptr(), s["v"].data_ptr(),
                               s["out"].data_ptr(), B, H, N, dk, dv, w["causal"], EPS, code,
                               None, None, ws.data_ptr(), ws.numel(), sp)
        assert st == 0, la.lib().la_last_error()
        if with_bwd:
            st = la.la_backward_saved(s["q"].data_ptr(), s["k"].data_ptr(), s["v"].data_ptr(),
                                      s["g"].data_ptr(), s["dq"].data_ptr(), s["dk"].data_ptr(),
                                      s["dv"].data_ptr(), B, H, N, dk, dv, w["causal"], EPS, code,
                                      ws.data_ptr(), ws.numel(), wsb.data_ptr(), wsb.numel(), sp)
            assert st == 0, la.lib().la_last_error()

    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    torch.cuda.synchronize()
    # warm the library's event pool outside capture
    la.la_profile_enable(1)
    with torch.cuda.stream(stream):
        for i in range(K):
            step(i)
    torch.cuda.synchronize()
    la.la_profile_enable(0)
    la.la_profile_read()
    ms, launches, _ = _graph_time(step, K, stream, barrier)
    _, _, spans = _graph_time(step, K, stream, lambda: None, profile=True)
    return dict(ms=ms, launches=launches, spans=_span_stats(spans), rotations=R,
                bytes_per_set=per_set)


def run_decode(w, K, W, barrier):
    import torch
    import causal_linear_attention_la_gb300 as la
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(w["seed"])
    B, H, dk, dv = w["B"], w["H"], w["dk"], w["dv"]
    p = w["prefill"]
    d = dk
    qp = (torch.randn((p["B"], p["H"], p["N"], d), generator=gen, device=dev) * d ** -0.5).to(torch.bfloat16)
    kp = (torch.randn((p["B"], p["H"], p["N"], d), generator=gen, device=dev) * d ** -0.5).to(torch.bfloat16)
    vp = (torch.randn((p["B"], p["H"], p["N"], d), generator=gen, device=dev) * d ** -0.5).to(torch.bfloat16)
    torch.cuda.synchronize()
    t0 = time.time()
    _, Sp, zp = la.forward(qp, kp, vp, return_state=True)
    torch.cuda.synchronize()
    prefill_s = time.time() - t0
    del qp, kp, vp
    src = torch.arange(B * H, device=dev) % p["H"]
    S = Sp[0][src].reshape(B, H, dk, dv).contiguous()
    z = zp[0][src].reshape(B, H, dk).contiguous()
    T = w["steps"]
    nt = w.get("tokens", 1)             # tokens per call
    qs = (torch.randn((T, B, H, nt, dk), generator=gen, device=dev) * dk ** -0.5).to(torch.bfloat16)
    ks = (torch.randn((T, B, H, nt, dk), generator=gen, device=dev) * dk ** -0.5).to(torch.bfloat16)
    vs = (torch.randn((T, B, H, nt, dv), generator=gen, device=dev) * dv ** -0.5).to(torch.bfloat16)
    out = torch.empty((T, B, H, nt, dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream()

    variant = w.get("variant")
    alpha = torch.linspace(0.9, 0.999, H, device=dev)       # per-head decay factors
    if variant == "delta":
        # unit-norm keys: each write replaces what its key held
        ks = ks / ks.float().norm(dim=-1, keepdim=True).to(ks.dtype)

    def step(i):
        sp = torch.cuda.current_stream().cuda_stream
        if variant == "decay":
            st = la.la_decode_steps_decay(S.data_ptr(), z.data_ptr(), qs[i].data_ptr(), ks[i].data_ptr(),
                                          vs[i].data_ptr(), out[i].data_ptr(), B, H, nt, dk, dv,
                                          alpha.data_ptr(), EPS, la.LA_BF16, sp)
        elif variant == "delta":
            st = la.la_decode_steps_delta(S.data_ptr(), qs[i].data_ptr(), ks[i].data_ptr(),
                                          vs[i].data_ptr(), out[i].data_ptr(), B, H, nt, dk, dv,
                                          la.LA_BF16, sp)
        elif nt == 1:
            st = la.la_decode_step(S.data_ptr(), z.data_ptr(), qs[i].data_ptr(), ks[i].data_ptr(),
                                   vs[i].data_ptr(), out[i].data_ptr(), B, H, dk, dv, EPS,
                                   la.LA_BF16, sp)
        else:
            st = la.la_decode_steps(S.data_ptr(), z.data_ptr(), qs[i].data_ptr(), ks[i].data_ptr(),
                                    vs[i].data_ptr(), out[i].data_ptr(), B, H, nt, dk, dv, EPS,
                                    la.LA_BF16, sp)
        assert st == 0, la.lib().la_last_error()

    with torch.cuda.stream(stream):
        for i in range(W):
            step(i % T)
    torch.cuda.synchronize()
    ms, launches, _ = _graph_time(step, T, stream, barrier)
    return dict(ms=ms, launches=launches, steps=T, prefill_s=prefill_s)


def run_delta_fwd(w, K, W, barrier):
    """K calls of la_forward_delta on one fp32 state, inputs rotating past L2
    (unit-norm keys: each write replaces what its key held)."""
    import torch
    import causal_linear_attention_la_gb300 as la
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(w["seed"])
    B, H, N, d = w["B"], w["H"], w["N"], w["dk"]
    R = _rotations(fwd_bytes(w))
    sets = []
    for _ in range(R):
        q = (torch.randn((B, H, N, d), generator=gen, device=dev) * d ** -0.5).to(torch.bfloat16)
        k = torch.randn((B, H, N, d), generator=gen, device=dev)
        k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        v = (torch.randn((B, H, N, d), generator=gen, device=dev) * d ** -0.5).to(torch.bfloat16)
        sets.append((q, k, v, torch.empty_like(v)))
    S = torch.zeros((B, H, d, d), device=dev)
    stream = torch.cuda.Stream()

    def step(i):
        q, k, v, o = sets[i % R]
        st = la.la_forward_delta(S.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 B, H, N, d, d, la.LA_BF16, torch.cuda.current_stream().cuda_stream)
        assert st == 0, la.lib().la_last_error()

    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    torch.cuda.synchronize()
    ms, launches, _ = _graph_time(step, K, stream, barrier)
    return dict(ms=ms, launches=launches, rotations=R, bytes_per_set=fwd_bytes(w))


def run_e2e(w, K, W, slices=E2E_SLICES):
    """Same forward metric through the host-buffer C-ABI call la_forward_host:
    per step the H2D copies of q, k, v from pinned host memory, the forward,
    and the D2H copy of out, timed with CUDA events on the calling stream.
    ``slices`` groups of sequences overlap their copies with the compute of
    their neighbours (1: copy, compute, copy in sequence)."""
    import torch
    import causal_linear_attention_la_gb300 as la
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    g = torch.Generator()
    g.manual_seed(w["seed"])
    hq = (torch.randn((B, H, N, dk), generator=g) * dk ** -0.5).to(torch.bfloat16).pin_memory()
    hk = (torch.randn((B, H, N, dk), generator=g) * dk ** -0.5).to(torch.bfloat16).pin_memory()
    hv = (torch.randn((B, H, N, dv), generator=g) * dv ** -0.5).to(torch.bfloat16).pin_memory()
    ho = torch.empty((B, H, N, dv), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(max(1, la.la_forward_host_workspace_size(B, H, N, dk, dv, w["causal"], la.LA_BF16, slices)),
                     dtype=torch.uint8, device="cuda")

    def step():
        la.forward_host(hq, hk, hv, causal=w["causal"], eps=EPS, out=ho, slices=slices, workspace=ws)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2
    d2h = ho.numel() * 2
    return dict(ms=ms, h2d=h2d, d2h=d2h, slices=slices)


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------


def _oracle_task(args):
    """One sequence of the oracle recurrence (runs in a pool worker)."""
    import oracle as orc
    q, k, v, causal, eps = args
    out = orc.forward_recurrent(q, k, v, causal=causal, eps=eps)
    return float(out[0, 0, -1, 0])


_POOL = None


def oracle_pool():
    """A process pool with one worker per host core, started with spawn (the
    workers import only numpy and the oracle; they never touch CUDA), warmed
    so that its start-up stays out of the timings. Returns (pool, workers)."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        try:
            cores = len(os.sched_getaffinity(0))
        except AttributeError:
            cores = os.cpu_count() or 1
        # one BLAS thread per worker: the pool provides the parallelism
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        pool = ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn"))
        z = np.zeros((1, 1, 2, 4), np.float32)
        list(pool.map(_oracle_task, [(z, z, z, True, EPS)] * cores))
        _POOL = (pool, cores)
    return _POOL


def oracle_sample(w, budget_s=10.0):
    """Time the fp64 oracle recurrence on a prefix of every sequence of the
    workload (one pool task per sequence, all host cores), growing the prefix
    until about ``budget_s`` of wall time. Returns (tokens/s, description,
    workers)."""
    from causal_linear_attention_la_gb300 import synth
    pool, cores = oracle_pool()
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    n = 32
    while True:
        q, k, v = synth.qkv(B, H, n, dk, dv, seed=w["seed"], dtype="bf16")
        tasks = [(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], w.get("causal", True), EPS)
                 for b in range(B) for h in range(H)]
        t0 = time.perf_counter()
        list(pool.map(_oracle_task, tasks))
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= N:
            break
        n = min(N, max(n * 2, int(n * budget_s / max(dt, 1e-3) * 0.9)))
    desc = (f"oracle recurrence (fp64 numpy), all {B}x{H} sequences, first {n} of {N} tokens, "
            f"one sequence per task over {cores} worker processes")
    return B * n / dt, desc, cores


def reference_arm(args, world, rank):
    if rank != 0:
        return 0
    w = WORKLOADS[MAIN]
    budget = args.ref_budget if args.ref_budget else max(1.0, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    desc = ""
    for i in range(args.warmup + args.steps):
        v, desc, threads = oracle_sample(w, budget_s=budget)
        if i >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals))
    tokens_per_step = w["B"] * w["N"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tokens_per_step / value, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": MAIN, **{k: w[k] for k in ("B", "H", "N", "dk", "dv", "causal")},
                   "eps": EPS, "note": "each step times the oracle on a bounded sample; "
                                       "value scaled to the whole batch's tokens"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sections", default="all", help="comma list of extra workloads or 'none'")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=None,
                    help="reference arm: seconds of oracle work per step (default: 60 s over all steps)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_env()

    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            rc = reference_arm(args, world, rank)
            dist.barrier()
            dist.destroy_process_group()
            return rc
        return reference_arm(args, world, rank)

    import torch
    import causal_linear_attention_la_gb300 as la
    from causal_linear_attention_la_gb300.build import build
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    barrier, max_over_ranks = dist_helpers(world, "cuda")
    if rank == 0:
        build()
    if world > 1:
        barrier()
    la.lib()
    peaks, peak_src = load_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    K, W = args.steps, args.warmup

    w = WORKLOADS[MAIN]
    r = run_forward(w, K, W, barrier)
    ms_total = max_over_ranks(r["ms"])
    tokens = w["B"] * w["N"] * K
    value = job_throughput(world, tokens, ms_total / 1e3)
    out_span = r["spans"].get("fwd_output", {"avg_ms": float("nan")})
    alg_bytes = fwd_bytes(w)
    achieved = alg_bytes / (out_span["avg_ms"] / 1e3) / 1e9
    e2e = run_e2e(w, K, W)
    e2e_ms = max_over_ranks(e2e["ms"])
    e2e_serial_ms = max_over_ranks(run_e2e(w, K, W, slices=1)["ms"])

    sections = {}
    wanted = list(WORKLOADS) if args.sections == "all" else (
        [] if args.sections == "none" else args.sections.split(","))
    for name in wanted:
        if name == MAIN or name not in WORKLOADS:
            continue
        ws = WORKLOADS[name]
        if ws["kind"] == "forward":
            rr = run_forward(ws, max(3, K // 5), W, barrier)
            kk = max(3, K // 5)
            t = max_over_ranks(rr["ms"]) / 1e3
            sp = rr["spans"].get("fwd_output", {"avg_ms": float("nan")})
            ach = fwd_bytes(ws) / (sp["avg_ms"] / 1e3) / 1e9
            sections[name] = {
                "value": job_throughput(world, ws["B"] * ws["N"] * kk, t), "unit": "tokens/s",
                "ms_per_step": 1e3 * t / kk, "steps": kk,
                "tflops_algorithmic": fwd_flops(ws) * kk / t / 1e12,
                "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": ach / peaks["hbm_gbs"], "kernel": "fwd_output",
                             "traffic": ncu_traffic("fwd_output_" + name)},
                "tensor": tensor_line(ws, sp["avg_ms"], peaks),
                "kernels": rr["spans"], "gpu_launches": rr["launches"],
                "l2": f"{rr['rotations']} input set(s) of {rr['bytes_per_set'] / 1e6:.0f} MB",
            }
        elif ws["kind"] == "decode":
            rr = run_decode(ws, K, W, barrier)
            t = max_over_ranks(rr["ms"]) / 1e3
            per = t / rr["steps"]
            nt = ws.get("tokens", 1)
            # the plain, decay-gated and delta-rule multi-token decodes take the tensor cores
            tc_decode = la.la_decode_path(ws["dk"], ws["dv"], la.LA_BF16, nt) == 1
            traffic_key = ("decodetc_" if tc_decode else "variants_" if ws.get("variant") else "decode_") + name
            # bytes of one call: the state once, q, k, v, out once per token
            call_bytes = decode_state_bytes(ws) + nt * decode_io_bytes(ws)
            gbs = decode_state_bytes(ws) / per / 1e9
            sections[name] = {
                "value": gbs, "unit": "GB/s (S/z traffic)", "ms_per_step": 1e3 * per,
                "steps": rr["steps"], "tokens_per_call": nt,
                "tokens_per_s": job_throughput(world, ws["B"] * nt, per),
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": gbs / peaks["hbm_gbs"],
                             "kernel": "decode_tc" if tc_decode else {"decay": "decay_tokens",
                                                                      "delta": "delta_tokens"}.get(
                                 ws.get("variant"), "decode"),
                             "traffic": ncu_traffic(traffic_key)},
                "bytes_per_step": call_bytes,
                "prefill_s_eager": rr["prefill_s"], "gpu_launches": rr["launches"],
                "l2": (f"state {decode_state_bytes(ws) / 2 / 1e6:.1f} MB, about the L2 "
                       f"({L2_BYTES / 1e6:.1f} MB): consecutive steps can meet the previous step's "
                       "lines in L2, so dram_frac counts measured DRAM bytes"),
            }
            dram = ncu_traffic(traffic_key)
            if dram is not None:
                sections[name]["dram_bytes_per_step"] = dram
                sections[name]["dram_gbs"] = dram / per / 1e9
                sections[name]["dram_frac"] = dram / per / 1e9 / peaks["hbm_gbs"]
        elif ws["kind"] == "delta_fwd":
            kk = max(3, K // 10)
            rr = run_delta_fwd(ws, kk, W, barrier)
            t = max_over_ranks(rr["ms"]) / 1e3
            mhz = sampler.summary()["sm_mhz"] or 2070.0
            ach = delta_flops(ws) * kk / t / 1e12
            # bf16 d = 128 with >= 64 heads runs the tensor-core group kernel
            tc = ws["dk"] == 128 and ws["B"] * ws["H"] >= 64
            peak = peaks["bf16_tflops"] if tc else fp32_peak_tflops(mhz)
            sections[name] = {
                "value": job_throughput(world, ws["B"] * ws["N"] * kk, t), "unit": "tokens/s",
                "ms_per_step": 1e3 * t / kk, "steps": kk,
                "roofline": {"bound": "tensor" if tc else "alu", "achieved": ach, "peak": peak,
                             "unit": "TFLOP/s", "frac": ach / peak,
                             "kernel": "decode_tc_delta" if tc else "delta_chunk",
                             "peak_source": (f"{peak_src} bf16_tflops" if tc else
                                             f"152 SMs x 128 fp32 FMA lanes x 2 at {mhz:.0f} MHz"),
                             "flops": "the token recurrence's 6 dk dv per token-head"},
                "gpu_launches": rr["launches"],
                "l2": f"{rr['rotations']} input set(s) of {rr['bytes_per_set'] / 1e6:.0f} MB",
            }
        elif ws["kind"] == "fwdbwd":
            kk = max(3, K // 5)
            rr = run_forward(ws, kk, W, barrier, with_bwd=True)
            t = max_over_ranks(rr["ms"]) / 1e3
            s1 = rr["spans"].get("bwd_sweep1", {"avg_ms": float("nan")})["avg_ms"]
            s2 = rr["spans"].get("bwd_sweep2", {"avg_ms": float("nan")})["avg_ms"]
            ach = bwd_bytes(ws) / ((s1 + s2) / 1e3) / 1e9
            sections[name] = {
                "value": job_throughput(world, ws["B"] * ws["N"] * kk, t), "unit": "tokens/s (fwd+bwd)",
                "ms_per_step": 1e3 * t / kk, "steps": kk,
                "tflops_algorithmic": 3 * fwd_flops(ws) * kk / t / 1e12,
                "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": ach / peaks["hbm_gbs"], "kernel": "bwd_sweep1+bwd_sweep2",
                             "traffic": ncu_traffic("bwd_" + name)},
                "kernels": rr["spans"], "gpu_launches": rr["launches"],
                "l2": f"{rr['rotations']} input set(s) of {rr['bytes_per_set'] / 1e6:.0f} MB",
            }
    sampler.stop()

    if rank == 0:
        cpu_v, cpu_desc, cpu_threads = oracle_sample(w, budget_s=args.cpu_budget)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": ms_total / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": MAIN, **{k: w[k] for k in ("B", "H", "N", "dk", "dv", "causal")},
                       "eps": EPS, "tokens_per_step": w["B"] * w["N"],
                       "l2": f"inputs rotate over {r['rotations']} sets of {r['bytes_per_set'] / 1e6:.0f} MB",
                       "timing": "K steps captured in one CUDA graph, CUDA events around its replay",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "tflops_algorithmic": world * fwd_flops(w) * K / (ms_total / 1e3) / 1e12,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": ncu_traffic("fwd_output_" + MAIN), "kernel": "fwd_output",
                         "peak_source": f"{peak_src} hbm_gbs",
                         "algorithmic_bytes_per_launch": alg_bytes},
            "tensor": tensor_line(w, out_span["avg_ms"], peaks),
            "kernels": r["spans"],
            "cpu_baseline": {"value": cpu_v, "unit": "tokens/s", "cores": cpu_threads,
                             "kind": "oracle", "sample": cpu_desc},
            "e2e": {"value": job_throughput(world, tokens, e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "call": f"la_forward_host, {e2e['slices']} sequence groups",
                    "unpipelined_value": job_throughput(world, tokens, e2e_serial_ms / 1e3)},
            "gpu_launches": r["launches"],
            "clocks": sampler.summary(),
            "path": {"forward": ["cuda-core", "tensor-core"][la.la_forward_path(w["dk"], w["dv"], la.LA_BF16)],
                     "backward": ["cuda-core", "tensor-core"][la.la_backward_path(w["dk"], w["dv"], la.LA_BF16)]},
            "sections": sections,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
