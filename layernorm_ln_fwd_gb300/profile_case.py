"""Run one workload's forward + backward a few times, for a profiler to attach to.

    python -m layernorm_ln_fwd_gb300.profile_case --workload bf16_8192x768 --iters 3
    python -m layernorm_ln_fwd_gb300.profile_case --workload f32_262144x1000 --rows 32768
    python -m layernorm_ln_fwd_gb300.profile_case --workload bdr_bf16_8192x768 --rows 65536
    python -m layernorm_ln_fwd_gb300.profile_case --workload bf16_8192x1280 --cols 2560

Workloads are the LayerNorm ones of ``synth.WORKLOADS`` and the other fused row operations
of ``synth.OP_WORKLOADS`` (RMSNorm, softmax, cross-entropy, the bias + dropout + residual
prologue, its mask regenerated or stored as bits), with the seeded synthetic inputs of ``synth`` (``--rows`` keeps the workload's
width, dtype and distributions and takes fewer or more rows, for captures that must stay
small or spill out of L2; ``--cols`` likewise takes another width for a LayerNorm workload);
backwards use a caller-owned workspace, as the benchmark does.
Nothing is checked.
"""
from __future__ import annotations

import argparse

import torch

import layernorm_ln_fwd_gb300 as ln
from layernorm_ln_fwd_gb300 import synth


def layernorm_case(name: str, rows: int, iters: int, cols: int = 0) -> None:
    w = synth.WORKLOADS[name]
    rows, cols = rows or w.rows, cols or w.cols
    inp = synth.make_inputs(rows, cols, w.dtype, seed=0, x=w.x, res=w.res, dy=w.dy,
                            gamma=w.gamma, beta=w.beta)
    d = {k: v.cuda() for k, v in inp.items()}
    ws = torch.zeros(ln.workspace_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    for _ in range(iters):
        out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], w.eps)
        ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd, workspace=ws)


def op_case(name: str, rows: int, iters: int) -> None:
    op = synth.OP_WORKLOADS[name]
    R, C, kind = rows or op["rows"], op["cols"], op["kind"]
    spread = {"softmax": 3.0, "xent": 2.0}.get(kind, 1.0)
    d = synth.make_inputs(R, C, op["dtype"], seed=0, device="cuda", x=("normal", 0.0, spread))
    ws = torch.zeros(ln.workspace_bytes(R, C), dtype=torch.uint8, device="cuda")
    if kind == "softmax":
        mask = synth.causal_mask(op["mask_rows"], C, op["dtype"], device="cuda")
    if kind == "xent":
        t = torch.randint(0, C, (R,), generator=torch.Generator(device="cuda").manual_seed(0),
                          device="cuda", dtype=torch.int32)
    if kind in ("bdr", "bdr_keep"):
        bias = (0.1 * d["beta"].float()).to(d["beta"].dtype)
        keep = (torch.empty(ln.dropout_keep_bytes(R, C), dtype=torch.uint8, device="cuda")
                if kind == "bdr_keep" else None)
    for i in range(iters):
        if kind == "rms":
            out, res_out, rrms = ln.rms_fwd(d["x"], d["res"], d["gamma"], 1e-5)
            ln.rms_bwd(d["dy"], res_out, d["gamma"], rrms, workspace=ws)
        elif kind == "softmax":
            y = ln.softmax_fwd(d["x"], mask, op["scale"])
            ln.softmax_bwd(d["dy"], y, op["scale"])
        elif kind == "xent":
            ln.xent(d["x"], t, op["alpha"], 1.0 / R)
        else:
            out, res_out, mean, rstd = ln.fwd_bias_dropout(d["x"], bias, d["res"], d["gamma"],
                                                           d["beta"], 1e-5, op["p"], 17, i,
                                                           keep=keep)
            ln.dropout_bwd(d["dy"], op["p"], 17, i, workspace=ws, keep=keep)


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=synth.BENCH_WORKLOAD,
                    choices=list(synth.WORKLOADS) + list(synth.OP_WORKLOADS))
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--rows", type=int, default=0, help="rows to use (default: the workload's)")
    ap.add_argument("--cols", type=int, default=0,
                    help="width of a LayerNorm workload (default: the workload's)")
    args = ap.parse_args()
    if args.workload in synth.WORKLOADS:
        layernorm_case(args.workload, args.rows, args.iters, args.cols)
    else:
        if args.cols:
            ap.error("--cols applies to the LayerNorm workloads")
        op_case(args.workload, args.rows, args.iters)
    torch.cuda.synchronize()
    print(f"ran {args.iters} iterations of {args.workload} ({args.rows or 'all'} rows)")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
