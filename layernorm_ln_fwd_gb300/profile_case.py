"""Run one workload's forward + backward a few times, for a profiler to attach to.

    python -m layernorm_ln_fwd_gb300.profile_case --workload bf16_8192x768 --iters 3

Inputs are the seeded synthetic ones of ``synth``; the backward uses a caller-owned
workspace, as the benchmark does.  Nothing is checked or printed but the kernel names.
"""
from __future__ import annotations

import argparse

import torch

import layernorm_ln_fwd_gb300 as ln
from layernorm_ln_fwd_gb300 import synth


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=synth.BENCH_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    d = {k: v.cuda() for k, v in synth.workload_inputs(args.workload, seed=0).items()}
    ws = torch.zeros(ln.workspace_bytes(w.rows, w.cols), dtype=torch.uint8, device="cuda")
    for _ in range(args.iters):
        out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], w.eps)
        ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd, workspace=ws)
    torch.cuda.synchronize()
    print(f"ran {args.iters} x fwd+bwd of {args.workload}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
