"""Parity of the fused residual-add + RMSNorm kernels (called through the C ABI) with the
float64 oracle ("GPU Performance from First Principles", section 6.1): every kernel family,
ragged and unaligned rows, no residual, constant and all-zero rows, full-size GPT-2-shaped
problems on every row, bitwise-repeatable dgamma, and the shared workspace left zero.
Tolerances are those of ``lnparity`` (rrms as rstd)."""
import numpy as np
import pytest
import torch

import layernorm_ln_fwd_gb300 as ln
import lnparity as P
import oracle
from layernorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = synth.EPS


@pytest.fixture(autouse=True)
def _auto_path():
    ln.force_path(ln.PATH_AUTO)
    yield
    ln.force_path(ln.PATH_AUTO)


def run_gpu(inp, has_res=True, workspace=None):
    d = P.to_device(inp)
    out, res_out, rrms = ln.rms_fwd(d["x"], d["res"] if has_res else None, d["gamma"], EPS)
    dx, dgamma = ln.rms_bwd(d["dy"], res_out, d["gamma"], rrms, workspace=workspace)
    torch.cuda.synchronize()
    return {"out": out, "res_out": res_out, "rrms": rrms, "dx": dx, "dgamma": dgamma}


def run_oracle(inp, has_res=True):
    io = P.io_of(inp["x"].dtype)
    f = oracle.rms_fwd(P.to64(inp["x"]), P.to64(inp["res"]) if has_res else None,
                       P.to64(inp["gamma"]), EPS, io=io)
    dy = P.to64(inp["dy"])
    b = oracle.rms_bwd(dy, f["res_out"], P.to64(inp["gamma"]), f["rrms"], io=io)
    shat = f["res_out"] * f["rrms"][:, None]
    allow = 36.0 * 2.0 ** -24 * np.sqrt(((dy * shat) ** 2).sum(axis=0))
    return {"out": f["out"], "res_out": f["res_out"], "rrms": f["rrms"], "dx": b["dx"],
            "dgamma": b["dgamma"], "_allow": allow}


def compare(gpu, ref, io):
    infos = []
    for name in ("out", "res_out", "rrms", "dx"):
        infos.append(P.compare(name, P.to64(gpu[name]), ref[name], io))
    infos.append(P.compare("dgamma", P.to64(gpu["dgamma"]), ref["dgamma"], io, extra=ref["_allow"]))
    if io == "bf16":
        np.testing.assert_array_equal(P.to64(gpu["res_out"]), ref["res_out"])
    return infos


COLS = [1, 3, 8, 32, 33, 128, 768, 1000, 1001, 1024, 1280, 2048, 4096, 8192, 16384]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", [1, 300])
def test_shapes_against_oracle(dtype, rows, cols):
    inp = synth.make_inputs(rows, cols, dtype, seed=rows * 7 + cols)
    compare(run_gpu(inp), run_oracle(inp), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", [ln.PATH_WARP, ln.PATH_BLOCK, ln.PATH_SCALAR])
@pytest.mark.parametrize("rows,cols", [(5, 64), (37, 768), (64, 1024), (19, 1000), (9, 4104)])
def test_every_kernel_family(dtype, path, rows, cols):
    if dtype == "bf16" and cols == 1000:
        cols = 1000 - 8
    ln.force_path(path)
    inp = synth.make_inputs(rows, cols, dtype, seed=11 + path)
    compare(run_gpu(inp), run_oracle(inp), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [768, 8192])
def test_without_residual(dtype, cols):
    inp = synth.make_inputs(33, cols, dtype, seed=3)
    gpu = run_gpu(inp, has_res=False)
    compare(gpu, run_oracle(inp, has_res=False), dtype)
    assert torch.equal(gpu["res_out"].cpu(), inp["x"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", [ln.PATH_WARP, ln.PATH_BLOCK, ln.PATH_SCALAR])
def test_constant_zero_and_outlier_rows(dtype, path):
    """Constant rows (r = 1/sqrt(c^2 + eps)), all-zero rows (r = eps^-1/2, out = 0) and rows
    with a value 1000 standard deviations out."""
    ln.force_path(path)
    rows, cols = 24, 768
    inp = synth.make_inputs(rows, cols, dtype, seed=21)
    td = synth.torch_dtype(dtype)
    x = inp["x"].float().clone()
    x[0:4] = torch.tensor([0.0, 1.5, -3.0, 1e4])[:, None]
    x[4:8, 0] = 1000.0
    x[8:12, cols // 2] = -1000.0
    res = inp["res"].float().clone()
    res[0:4] = 0.0
    inp["x"], inp["res"] = x.to(td), res.to(td)
    gpu = run_gpu(inp)
    compare(gpu, run_oracle(inp), dtype)
    assert torch.count_nonzero(gpu["out"][0]) == 0
    np.testing.assert_allclose(P.to64(gpu["rrms"][0:1]), [EPS ** -0.5], rtol=5e-7)


@pytest.mark.parametrize("dtype,rows,cols", [("bf16", 8192, 768), ("bf16", 8192, 1280),
                                             ("f32", 4096, 1000), ("bf16", 4096, 8192),
                                             ("bf16", 2503, 1600), ("bf16", 2503, 2560),
                                             ("bf16", 2503, 4096), ("f32", 2503, 1600)])
def test_full_size_every_row_and_bitwise_repeatable(dtype, rows, cols):
    inp = synth.make_inputs(rows, cols, dtype, seed=0)
    gpu = run_gpu(inp)
    infos = compare(gpu, run_oracle(inp), dtype)
    assert all(i["n_over_stated"] == 0 for i in infos), infos
    d = P.to_device(inp)
    for _ in range(2):
        dx2, dg2 = ln.rms_bwd(d["dy"], gpu["res_out"], d["gamma"], gpu["rrms"])
        torch.cuda.synchronize()
        assert torch.equal(dg2, gpu["dgamma"]) and torch.equal(dx2, gpu["dx"])


def test_workspace_shared_with_layernorm_is_left_zero():
    """One caller-owned workspace serves RMSNorm and LayerNorm backwards in turn; each call
    leaves every byte zero (the RMSNorm writes one statistic's partial sums, not two)."""
    cases = [("bf16", 300, 768, ln.PATH_AUTO), ("f32", 300, 1024, ln.PATH_AUTO),
             ("bf16", 9, 4104, ln.PATH_BLOCK), ("f32", 7, 1001, ln.PATH_SCALAR)]
    ws = torch.zeros(max(ln.workspace_bytes(r, c) for _, r, c, _ in cases), dtype=torch.uint8,
                     device="cuda")
    for i, (dtype, rows, cols, path) in enumerate(cases):
        ln.force_path(path)
        inp = synth.make_inputs(rows, cols, dtype, seed=60 + i)
        compare(run_gpu(inp, workspace=ws), run_oracle(inp), dtype)
        assert int(torch.count_nonzero(ws)) == 0, (dtype, rows, cols, path)
        P.compare_all(P.run_gpu(inp, EPS, workspace=ws), P.run_oracle(inp, EPS), dtype,
                      conditioned=True)
        assert int(torch.count_nonzero(ws)) == 0, (dtype, rows, cols, path)


def test_launch_count():
    inp = synth.make_inputs(64, 768, "bf16", seed=10)
    d = P.to_device(inp)
    out, res_out, rrms = ln.rms_fwd(d["x"], d["res"], d["gamma"], EPS)
    assert ln.last_launch_count() == 1
    ln.rms_bwd(d["dy"], res_out, d["gamma"], rrms)
    assert ln.last_launch_count() == 1
