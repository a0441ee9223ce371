"""Parity with the float64 oracle on rows that stress the forward's row statistics, for every
kernel family (warp per row, block per row, scalar), with the bare stated tolerances (no
conditioning term):

* rows whose FIRST stored value (or a value elsewhere) is an outlier 10, 100 or 1000
  standard deviations from the rest: the statistics must not depend on which value comes
  first;
* x ~ N(10^4, 1), the cancellation case of "Accelerating Transformer on GPU (I)", section
  4.2, where E[x^2] - E[x]^2 in fp32 gives a variance <= 0;
* constant rows (variance 0: rstd = eps^-1/2, out = beta, xhat = 0).

The forward is compared as computed on both sides.  The backward is fed the same stored
inputs on both sides (the oracle forward's res_out, and its mean and rstd rounded to fp32,
the API's storage type), so that it is compared on its own arithmetic: with an fp32 mean of
10^4 the mean's own rounding (half an ulp, 5e-4) moves xhat by more than the fp32 tolerance,
which no kernel can avoid once the mean is stored in fp32.
"""
import numpy as np
import pytest
import torch

import layernorm_ln_fwd_gb300 as ln
import lnparity as P
import oracle
from layernorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = synth.EPS
FWD = ("out", "res_out", "mean", "rstd")


@pytest.fixture(autouse=True)
def _auto_path():
    ln.force_path(ln.PATH_AUTO)
    yield
    ln.force_path(ln.PATH_AUTO)


def _forward_bare(inp, has_res=True):
    gpu = P.run_gpu(inp, EPS, has_res=has_res)
    ref = P.run_oracle(inp, EPS, has_res=has_res)
    infos = P.compare_all({k: gpu[k] for k in FWD if k in gpu},
                          {k: ref[k] for k in FWD}, P.io_of(inp["x"].dtype))
    assert all(i["n_over_stated"] == 0 for i in infos), infos
    return gpu


def _backward_on_stored(inp, has_res=True, rounding_allowance=False):
    """The backward alone on the oracle forward's stored res_out, mean and rstd.

    ``rounding_allowance``: add to dx's bound the fp32 rounding of g and of the row sums as
    rstd amplifies it, 4 * 2^-24 * rstd * (|g| + |sum g| / n).  It matters only where rstd
    is huge (a constant row: rstd = eps^-1/2 ~ 316, so one rounding of a g ~ 1 becomes
    ~2e-5 of dx): no fp32 arithmetic can do better there."""
    io = P.io_of(inp["x"].dtype)
    td = inp["x"].dtype
    f = oracle.ln_fwd(P.to64(inp["x"]), P.to64(inp["res"]) if has_res else None,
                      P.to64(inp["gamma"]), P.to64(inp["beta"]), EPS, io=io, want_out=False)
    mean32 = oracle.round_io(f["mean"], "f32")
    rstd32 = oracle.round_io(f["rstd"], "f32")
    dev = lambda a, t=td: torch.tensor(a).to(t).cuda()  # noqa: E731  (exact casts)
    dx, dg, db = ln.bwd(inp["dy"].cuda(), dev(f["res_out"]), inp["gamma"].cuda(),
                        dev(mean32, torch.float32), dev(rstd32, torch.float32))
    torch.cuda.synchronize()
    b = oracle.ln_bwd(P.to64(inp["dy"]), f["res_out"], P.to64(inp["gamma"]), mean32, rstd32,
                      io=io)
    extra_dx = None
    if rounding_allowance and io == "f32":
        g64 = P.to64(inp["gamma"])[None, :] * P.to64(inp["dy"])
        extra_dx = 4 * 2.0 ** -24 * rstd32[:, None] * (
            np.abs(g64) + np.abs(g64.sum(axis=1, keepdims=True)) / g64.shape[1])
    for name, g in (("dx", dx), ("dgamma", dg), ("dbeta", db)):
        info = P.compare(name, P.to64(g), b[name], io, extra=extra_dx if name == "dx" else None)
        if not (name == "dx" and extra_dx is not None):
            assert info["n_over_stated"] == 0


# (path, dtype, cols): every kernel family, including rows that are not a multiple of the
# 32-lane vector stride (1000 fp32, 1032 bf16) and rows that need a scalar kernel (1001).
CASES = [
    (ln.PATH_WARP, "f32", 768), (ln.PATH_WARP, "bf16", 768), (ln.PATH_WARP, "f32", 1000),
    (ln.PATH_WARP, "bf16", 1280), (ln.PATH_WARP, "bf16", 1032), (ln.PATH_AUTO, "bf16", 2560),
    (ln.PATH_BLOCK, "f32", 4104), (ln.PATH_BLOCK, "bf16", 8192), (ln.PATH_BLOCK, "bf16", 768),
    (ln.PATH_BLOCK, "f32", 1000),
    (ln.PATH_SCALAR, "f32", 1001), (ln.PATH_SCALAR, "bf16", 768), (ln.PATH_SCALAR, "f32", 2048),
]


def _outlier_inputs(dtype, rows, cols, seed):
    """x, res ~ N(0, 1) (s = x + res has sigma = sqrt 2); row r gets one value k sigma from
    the rest, k in {10, 100, 1000} with both signs, in column 0 for most rows and in the
    middle or last column for some; every seventh row is left as drawn."""
    inp = synth.make_inputs(rows, cols, dtype, seed=seed)
    x = inp["x"].float().clone()
    res = inp["res"].float().clone()
    ks = [10.0, 100.0, 1000.0]
    for r in range(rows):
        if r % 7 == 6:
            continue
        k = ks[r % 3] * (1.0 if (r // 3) % 2 == 0 else -1.0)
        col = 0 if r % 5 else (cols // 2 if r % 10 else cols - 1)
        x[r, col] = k * 2.0 ** 0.5
        res[r, col] = 0.0
    td = synth.torch_dtype(dtype)
    inp["x"], inp["res"] = x.to(td), res.to(td)
    return inp


@pytest.mark.parametrize("path,dtype,cols", CASES)
def test_outlier_rows(path, dtype, cols):
    ln.force_path(path)
    inp = _outlier_inputs(dtype, 84, cols, seed=cols + path)
    _forward_bare(inp)
    _backward_on_stored(inp)


@pytest.mark.parametrize("path,dtype,cols", CASES)
def test_large_mean_rows(path, dtype, cols):
    """x ~ N(10^4, 1), res ~ N(0, 1).  In bf16 the values near 10^4 are 64 apart, so most
    rows hold two or three distinct values: also a near-constant case."""
    ln.force_path(path)
    inp = synth.make_inputs(50, cols, dtype, seed=cols + 11 * path, x=("normal", 1e4, 1.0))
    _forward_bare(inp)
    _backward_on_stored(inp)


@pytest.mark.parametrize("path,dtype,cols", CASES + [(ln.PATH_WARP, "bf16", 8),
                                                     (ln.PATH_WARP, "f32", 4),
                                                     (ln.PATH_SCALAR, "f32", 2)])
def test_constant_rows(path, dtype, cols):
    """Every row constant (values whose row sums are exact, so the oracle's mean and the
    GPU's are the same number): var = 0, rstd = eps^-1/2, out = beta, xhat = 0, dgamma = 0,
    dx = rstd (g - mean(g)).  The forward and dgamma, dbeta are held to the bare stated
    bound; fp32 dx adds the rounding allowance of ``_backward_on_stored``."""
    ln.force_path(path)
    rows = 40
    vals = torch.tensor([0.0, 1.0, -3.5, 0.75, 1000.0, -2.0 ** 20, 96.0, 1e4])
    inp = synth.make_inputs(rows, cols, dtype, seed=cols + 3)
    td = synth.torch_dtype(dtype)
    inp["x"] = vals[torch.arange(rows) % len(vals)][:, None].expand(rows, cols).to(td).contiguous()
    inp["res"] = torch.zeros(rows, cols, dtype=td)
    gpu = _forward_bare(inp)
    # out is beta exactly (rounded once from beta itself) and rstd is eps^-1/2.
    assert torch.equal(gpu["out"].cpu(), inp["beta"][None, :].expand(rows, cols))
    np.testing.assert_allclose(P.to64(gpu["rstd"]), EPS ** -0.5, rtol=5e-7)
    _backward_on_stored(inp, rounding_allowance=True)
    # Without a residual (plain LayerNorm of x) as well.
    _forward_bare(inp, has_res=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_statistics_do_not_depend_on_column_order(dtype):
    """Rotating every row by one column (the first value moves to the end) changes which
    value the kernels shift by: mean and rstd must stay within the stated tolerance of each
    other and of the oracle on both orders."""
    inp = _outlier_inputs(dtype, 84, 768, seed=5)
    a = _forward_bare(inp)
    rot = dict(inp)
    rot["x"] = torch.roll(inp["x"], shifts=-1, dims=1).contiguous()
    rot["res"] = torch.roll(inp["res"], shifts=-1, dims=1).contiguous()
    rot["gamma"] = torch.roll(inp["gamma"], shifts=-1).contiguous()
    rot["beta"] = torch.roll(inp["beta"], shifts=-1).contiguous()
    b = _forward_bare(rot)
    for k in ("mean", "rstd"):
        P.compare(k, P.to64(b[k]), P.to64(a[k]).astype(np.float64), "f32")
