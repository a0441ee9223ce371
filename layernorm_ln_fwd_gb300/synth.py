"""Seeded synthetic inputs for the fused residual-add + LayerNorm workloads.

This module holds random draws only -- none of the method's arithmetic -- so that the CUDA
path and the float64 oracle can be fed identical inputs without sharing any code.

Recipe (every workload): a CPU ``torch.Generator`` seeded with ``seed`` draws, in this order,
x, res, dy (each [rows, cols]), gamma and beta ([cols]) as float32 from the stated
distributions; each tensor is then cast to the I/O dtype (bf16 casts round to nearest even).
gamma ~ N(1, 0.1), beta ~ N(0, 0.1) and eps = 1e-5 in every workload.

The shapes follow the Transformer shapes on the pages: 8 sequences x 1024 tokens with
hidden size 768 (GPT-2 small, the width llm.c uses) and 1280 (GPT-2 large, the shape the
whole-step accounting in "Accelerating Transformer on GPU (II): Training with LightSeq2",
section 1.2, uses), plus a wide-row case with a large mean (the cancellation experiment of
"Accelerating Transformer on GPU (I)", section 4.2) and a large fp32 case whose width is
not a multiple of the 128-column warp stride.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

EPS = 1e-5


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str  # "f32" or "bf16": the I/O (storage) dtype; arithmetic is fp32
    rows: int
    cols: int
    x: tuple = ("normal", 0.0, 1.0)
    res: tuple = ("normal", 0.0, 1.0)
    dy: tuple = ("normal", 0.0, 1.0)
    gamma: tuple = ("normal", 1.0, 0.1)
    beta: tuple = ("normal", 0.0, 0.1)
    eps: float = EPS
    note: str = field(default="", compare=False)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("f32_64x768", "f32", 64, 768,
                 note="small fp32 case the oracle finishes in well under a second"),
        Workload("bf16_8192x768", "bf16", 8192, 768,
                 note="GPT-2 small shape: 8 x 1024 tokens, hidden 768"),
        Workload("bf16_8192x1280", "bf16", 8192, 1280,
                 note="GPT-2 large shape: 8 x 1024 tokens, hidden 1280"),
        Workload("bf16_4096x8192_mean100", "bf16", 4096, 8192, x=("normal", 100.0, 1.0),
                 note="wide rows; x has mean 100 (stresses E[x^2]-E[x]^2 cancellation)"),
        Workload("f32_262144x1000", "f32", 262144, 1000, x=("uniform", -3.0, 3.0),
                 res=("normal", 0.0, 0.5),
                 note="large fp32 case, 1000 columns: ragged against the warp stride"),
    ]
}

# The workload of the benchmark's headline line: the largest one (every workload is also
# timed, in the same line).
BENCH_WORKLOAD = "f32_262144x1000"

# Other Transformer widths, timed in the benchmark's line beside the workloads above (not
# benchmark configurations): rows wider than one warp's registers, which take the tile
# kernels with 2 or 4 warps per row.
EXTRA_WORKLOADS = {
    w.name: w
    for w in [
        Workload("bf16_8192x1600", "bf16", 8192, 1600,
                 note="GPT-2 XL hidden size 1600: 2 warps per row in the backward"),
        Workload("bf16_8192x2560", "bf16", 8192, 2560,
                 note="4 warps per row in the forward and the backward"),
        Workload("f32_8192x1280", "f32", 8192, 1280,
                 note="fp32 rows of 1280 columns: 2 warps per row in the backward"),
    ]
}


def workload(name: str) -> Workload:
    """A workload of either table."""
    return WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]


def torch_dtype(dtype: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def _draw(gen: torch.Generator, shape, dist, device="cpu") -> torch.Tensor:
    kind, a, b = dist
    if kind == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32, device=device) * b + a
    if kind == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32, device=device) * (b - a) + a
    if kind == "int":  # integers drawn uniformly from [a, b]
        return torch.randint(int(a), int(b) + 1, shape, generator=gen,
                             device=device).to(torch.float32)
    if kind == "const":
        return torch.full(shape, float(a), dtype=torch.float32, device=device)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(rows: int, cols: int, dtype: str, seed: int = 0, x=("normal", 0.0, 1.0),
                res=("normal", 0.0, 1.0), dy=("normal", 0.0, 1.0), gamma=("normal", 1.0, 0.1),
                beta=("normal", 0.0, 0.1), device="cpu") -> dict:
    """Tensors in the I/O dtype: x, res, dy [rows, cols]; gamma, beta [cols].

    With the default ``device="cpu"`` the draws come from a CPU generator (the tests' inputs,
    identical on every machine).  Another device draws with that device's own seeded
    generator: the same distributions from a different random stream, for the benchmark's
    large buffer sets."""
    gen = torch.Generator(device=device).manual_seed(int(seed))
    td = torch_dtype(dtype)
    out = {}
    for name, shape, dist in (("x", (rows, cols), x), ("res", (rows, cols), res),
                              ("dy", (rows, cols), dy), ("gamma", (cols,), gamma),
                              ("beta", (cols,), beta)):
        out[name] = _draw(gen, shape, dist, device).to(td).contiguous()
    return out


def workload_inputs(name: str, seed: int = 0, device="cpu") -> dict:
    w = workload(name)
    return make_inputs(w.rows, w.cols, w.dtype, seed=seed, x=w.x, res=w.res, dy=w.dy,
                       gamma=w.gamma, beta=w.beta, device=device)


# Workloads of the other fused row operations (the pages' shapes):
#  * fused add + RMSNorm ("GPU Performance from First Principles", section 6.1) at the two
#    GPT-2 LayerNorm shapes above, same distributions (no beta);
#  * fused softmax of attention scores, batch x heads x L rows of L columns with a causal
#    mask and the 1/sqrt(64) scale: 8 x 16 x 512 x 512 ("Accelerating Transformer on GPU
#    (II)", section 3.2) and 2 x 16 x 256 x 256 ("... (I)", section 4.1); scores ~ N(0, 3),
#    dy ~ N(0, 1).
OP_WORKLOADS = {
    "rms_bf16_8192x768": dict(kind="rms", dtype="bf16", rows=8192, cols=768),
    "rms_bf16_8192x1280": dict(kind="rms", dtype="bf16", rows=8192, cols=1280),
    "softmax_bf16_65536x512_causal": dict(kind="softmax", dtype="bf16", rows=65536, cols=512,
                                          mask_rows=512, scale=0.125),
    "softmax_bf16_8192x256_causal": dict(kind="softmax", dtype="bf16", rows=8192, cols=256,
                                         mask_rows=256, scale=0.125),
    # fused cross-entropy of GPT-2 small's classifier: 8 x 1024 tokens over llm.c's padded
    # vocabulary of 50304 ("llm.c: the llmc/ CUDA kernel layer", section 6), logits ~ N(0, 2),
    # label smoothing 0.1 ("Accelerating Transformer on GPU (I)", section 5.2), mean loss.
    "xent_bf16_8192x50304": dict(kind="xent", dtype="bf16", rows=8192, cols=50304, alpha=0.1),
    # bias + dropout + residual prologue of the LayerNorm forward at the GPT-2 small shape,
    # p = 0.1 ("Accelerating Transformer on GPU (I)", section 2.3).
    "bdr_bf16_8192x768": dict(kind="bdr", dtype="bf16", rows=8192, cols=768, p=0.1),
    # the same with the keep decisions stored as bits by the forward, read by the backward
    "bdr_keep_bf16_8192x768": dict(kind="bdr_keep", dtype="bf16", rows=8192, cols=768, p=0.1),
}


def causal_mask(L: int, cols: int, dtype: str, device="cpu") -> torch.Tensor:
    """[L, cols] additive mask: query q keeps keys k <= q * cols / L (0), the rest -inf."""
    q = torch.arange(L, device=device)[:, None]
    k = torch.arange(cols, device=device)[None, :]
    m = torch.zeros(L, cols, device=device)
    m[k > q * cols // L] = float("-inf")
    return m.to(torch_dtype(dtype))
