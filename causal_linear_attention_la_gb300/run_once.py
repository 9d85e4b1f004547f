"""Run a few calls of one workload on random inputs (for profilers).

    python -m causal_linear_attention_la_gb300.run_once --workload fwd --B 4 --H 8 --N 4096 --d 64 --calls 2

Workloads: fwd (la_forward; la_forward_decay with --decay; la_forward_delta,
the chunked delta rule on unit-norm keys, with --delta), bwd (la_forward
then la_backward), decode (la_decode_step on zero-initialised states, or
la_decode_steps with --tokens T; --variant decay|delta for the gated and
delta-rule updates). Inputs are seeded normal values scaled by 1/sqrt(d),
bf16 unless --f32; decay factors 0.9 .. 0.999 over the heads.
"""

import argparse
import sys

import torch

import causal_linear_attention_la_gb300 as la


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=["fwd", "bwd", "decode"], default="fwd")
    ap.add_argument("--B", type=int, default=4)
    ap.add_argument("--H", type=int, default=8)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--d", type=int, default=64)
    ap.add_argument("--calls", type=int, default=2)
    ap.add_argument("--tokens", type=int, default=1, help="decode: tokens per call (la_decode_steps when > 1)")
    ap.add_argument("--noncausal", action="store_true")
    ap.add_argument("--decay", action="store_true", help="fwd: decay-gated forward")
    ap.add_argument("--delta", action="store_true", help="fwd: chunked delta rule")
    ap.add_argument("--variant", choices=["plain", "decay", "delta"], default="plain",
                    help="decode: state update variant")
    ap.add_argument("--f32", action="store_true")
    args = ap.parse_args(argv)
    from causal_linear_attention_la_gb300.build import build
    build()
    dt = torch.float32 if args.f32 else torch.bfloat16
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    B, H, N, d = args.B, args.H, args.N, args.d

    def rnd(*shape, scale=d ** -0.5):
        return (torch.randn(shape, generator=g, device="cuda") * scale).to(dt)

    causal = not args.noncausal
    alpha = torch.linspace(0.9, 0.999, H, device="cuda")
    if args.workload == "decode":
        S = torch.zeros((B, H, d, d), device="cuda")
        z = torch.zeros((B, H, d), device="cuda")
        if args.variant != "plain":
            T = args.tokens
            q, k, v = rnd(B, H, T, d), rnd(B, H, T, d), rnd(B, H, T, d)
            for _ in range(args.calls):
                if args.variant == "decay":
                    la.decode_steps_decay(S, z, q, k, v, alpha)
                else:
                    la.decode_steps_delta(S, q, k, v)
        elif args.tokens > 1:
            T = args.tokens
            q, k, v = rnd(B, H, T, d), rnd(B, H, T, d), rnd(B, H, T, d)
            for _ in range(args.calls):
                la.decode_steps(S, z, q, k, v)
        else:
            q, k, v = rnd(B, H, d), rnd(B, H, d), rnd(B, H, d)
            for _ in range(args.calls):
                la.decode_step(S, z, q, k, v)
    else:
        q, k, v = rnd(B, H, N, d), rnd(B, H, N, d), rnd(B, H, N, d)
        gout = rnd(B, H, N, d, scale=1.0)
        if args.delta:
            k = (k.float() / k.float().norm(dim=-1, keepdim=True)).to(dt)
            S = torch.zeros((B, H, d, d), device="cuda")
        for _ in range(args.calls):
            if args.delta:
                la.forward_delta(S, q, k, v)
            elif args.decay:
                la.forward_decay(q, k, v, alpha)
            else:
                la.forward(q, k, v, causal=causal)
            if args.workload == "bwd":
                la.backward(q, k, v, gout, causal=causal)
    torch.cuda.synchronize()
    st = la.la_device_status(True)
    print(f"done: {args.workload} B={B} H={H} N={N} d={d} calls={args.calls} status={st}")
    return 0 if st == la.LA_OK else 1


if __name__ == "__main__":
    sys.exit(main())
