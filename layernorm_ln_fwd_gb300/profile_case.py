"""Run one workload's forward + backward a few times, for a profiler to attach to.

    python -m layernorm_ln_fwd_gb300.profile_case --workload bf16_8192x768 --iters 3
    python -m layernorm_ln_fwd_gb300.profile_case --workload f32_262144x1000 --rows 32768

Inputs are the seeded synthetic ones of ``synth`` (``--rows`` keeps the workload's width,
dtype and distributions and takes fewer rows, for captures that must stay small); the
backward uses a caller-owned workspace, as the benchmark does.  Nothing is checked.
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
    ap.add_argument("--rows", type=int, default=0, help="rows to use (default: the workload's)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    rows = args.rows or w.rows
    inp = synth.make_inputs(rows, w.cols, w.dtype, seed=0, x=w.x, res=w.res, dy=w.dy,
                            gamma=w.gamma, beta=w.beta)
    d = {k: v.cuda() for k, v in inp.items()}
    ws = torch.zeros(ln.workspace_bytes(rows, w.cols), dtype=torch.uint8, device="cuda")
    for _ in range(args.iters):
        out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], w.eps)
        ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd, workspace=ws)
    torch.cuda.synchronize()
    print(f"ran {args.iters} x fwd+bwd of {args.workload} ({rows} rows)")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
