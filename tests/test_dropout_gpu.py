"""Parity of the bias + dropout + residual prologue of the LayerNorm forward ("Accelerating
Transformer on GPU (I)", section 2.3) and of its backward with the float64 oracle.

The dropout decisions are integers on both sides (Philox-4x32-10 words against the same
threshold), so the mask must agree exactly: a dropped element's res_out is its residual, bit
for bit.  A kept element's res_out = res + (h + bias) / (1 - p) is held to one unit in the
last place of the I/O type (fp32: the stated 2e-5) plus the error of the fp32 intermediate:
1 / (1 - p) is not a machine number, the kernel forms t = (h + bias) * fp32(1 / (1 - p)) and
res + t in fp32 (at most 4 fp32 roundings of |t|, delta = 4 * 2^-24 * |t|), and that value can
sit on the other side of an I/O rounding boundary from the exact one.  Where res and t cancel
(the exact sum 0, the fp32 one 2^-26) only delta bounds the difference.  The LayerNorm of
res_out is compared with the oracle's LayerNorm of the GPU's res_out at the bare stated
tolerances.  The backward's dh and dbias are compared with the
oracle's on the same ds.
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


@pytest.fixture(autouse=True)
def _auto_path():
    ln.force_path(ln.PATH_AUTO)
    yield
    ln.force_path(ln.PATH_AUTO)


def one_ulp(v, io):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - (23 if io == "f32" else 7))


def run(rows, cols, dtype, p, seed, offset, path=ln.PATH_AUTO, check_bwd=True):
    ln.force_path(path)
    inp = synth.make_inputs(rows, cols, dtype, seed=rows + cols)
    bias = synth.make_inputs(1, cols, dtype, seed=3, x=("normal", 0.0, 0.1))["x"][0]
    d = P.to_device(inp)
    out, res_out, mean, rstd = ln.fwd_bias_dropout(d["x"], bias.cuda(), d["res"], d["gamma"],
                                                   d["beta"], EPS, p, seed, offset)
    torch.cuda.synchronize()
    io = dtype
    keep = oracle.dropout_mask(seed, offset, p, rows, cols).astype(bool)
    ref = oracle.bdr_ln_fwd(P.to64(inp["x"]), P.to64(bias), P.to64(inp["res"]),
                            P.to64(inp["gamma"]), P.to64(inp["beta"]), EPS, p, seed, offset, io=io)
    g_res = P.to64(res_out)
    # The mask: dropped elements carry the residual itself.
    np.testing.assert_array_equal(g_res[~keep], P.to64(inp["res"])[~keep])
    err = np.abs(g_res - ref["res_out"])
    t = np.abs(P.to64(inp["x"]) + P.to64(bias)[None, :]) / (1 - p)
    delta = 4.0 * 2.0 ** -24 * t
    tol = np.maximum(one_ulp(np.abs(ref["res_out"]) + delta, io), 2e-5 if io == "f32" else 0.0) + delta
    assert np.all(err <= tol), float(err.max())
    # The LayerNorm of what the prologue stored.
    f = oracle.ln_fwd(g_res, None, P.to64(inp["gamma"]), P.to64(inp["beta"]), EPS, io=io)
    for name, g in (("out", out), ("mean", mean), ("rstd", rstd)):
        info = P.compare(name, P.to64(g), f[name], io)
        assert info["n_over_stated"] == 0
    if not check_bwd:
        return
    # Backward of the prologue on the LayerNorm backward's dx.
    ds, _, _ = ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd)
    dh, dbias = ln.dropout_bwd(ds, p, seed, offset)
    torch.cuda.synchronize()
    b = oracle.dropout_bwd(P.to64(ds), p, seed, offset, io=io)
    P.compare("dx", P.to64(dh), b["dh"], io)
    terms = keep * P.to64(ds) / (1 - p)
    allow = 36.0 * 2.0 ** -24 * np.sqrt((terms ** 2).sum(axis=0))
    P.compare("dbeta", P.to64(dbias), b["dbias"], io, extra=allow)
    # Repeatable bit for bit.
    dh2, dbias2 = ln.dropout_bwd(ds, p, seed, offset)
    torch.cuda.synchronize()
    assert torch.equal(dh2, dh) and torch.equal(dbias2, dbias)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(1, 8), (7, 768), (300, 1000), (300, 1001), (64, 1280),
                                       (9, 4104), (5, 8192)])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_shapes(dtype, rows, cols, p):
    if dtype == "bf16" and cols == 1000:
        cols = 1000 - 8
    run(rows, cols, dtype, p, seed=11, offset=rows)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", [ln.PATH_WARP, ln.PATH_BLOCK, ln.PATH_SCALAR])
def test_every_kernel_family(dtype, path):
    run(37, 768, dtype, 0.3, seed=2 ** 40 + 5, offset=2 ** 33 + 1, path=path, check_bwd=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_probability_is_the_fused_residual_layernorm(dtype):
    inp = synth.make_inputs(50, 768, dtype, seed=1)
    d = P.to_device(inp)
    zero = torch.zeros(768, dtype=d["x"].dtype, device="cuda")
    a = ln.fwd_bias_dropout(d["x"], zero, d["res"], d["gamma"], d["beta"], EPS, 0.0, 1, 2)
    b = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], EPS)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1])  # res + x: the same rounding of an exact sum
    if dtype == "bf16":
        for k in (0, 2, 3):
            assert torch.equal(a[k], b[k])


def test_full_size_gpt2_small():
    run(8192, 768, "bf16", 0.1, seed=1234, offset=0)


def test_workspace_left_zero_and_shared_with_the_backward():
    rows, cols = 300, 768
    ws = torch.zeros(ln.workspace_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    inp = synth.make_inputs(rows, cols, "bf16", seed=4)
    d = P.to_device(inp)
    for _ in range(2):
        ln.bwd(d["dy"], d["x"], d["gamma"], torch.zeros(rows, device="cuda"),
               torch.ones(rows, device="cuda"), workspace=ws)
        ln.dropout_bwd(d["dy"], 0.2, 5, 6, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws)) == 0


def test_invalid_arguments():
    x = torch.zeros(4, 8, device="cuda")
    b = torch.zeros(8, device="cuda")
    with pytest.raises(ln.LnError):
        ln.fwd_bias_dropout(x, b, x, b, b, EPS, 1.0, 0, 0)
    with pytest.raises(ln.LnError):
        ln.dropout_bwd(x, -0.1, 0, 0)


# ---------------------------------------------------------------------------------------
# The keep decisions stored as bits by the forward and read by the backward.

def oracle_keep_bytes(seed, offset, p, rows, cols):
    """The oracle's mask packed as the library stores it: bit (c % 8) of byte
    [row, c // 8], rows padded to whole bytes with zero bits."""
    m = oracle.dropout_mask(seed, offset, p, rows, cols).astype(np.uint8)
    return np.packbits(m, axis=1, bitorder="little")


@pytest.mark.parametrize("dtype,rows,cols,path", [
    ("bf16", 300, 768, ln.PATH_AUTO),      # warp per row
    ("bf16", 37, 4104, ln.PATH_AUTO),      # block per row
    ("bf16", 300, 1001, ln.PATH_AUTO),     # scalar (not 16-byte rows)
    ("bf16", 5, 8, ln.PATH_AUTO),          # one vector per row
    ("f32", 64, 1000, ln.PATH_AUTO),       # fp32: two lanes share a byte
    ("f32", 7, 1004, ln.PATH_AUTO),        # an odd number of vectors per row
    ("f32", 9, 4104, ln.PATH_AUTO),        # fp32 block per row
    ("f32", 37, 768, ln.PATH_BLOCK),
    ("bf16", 37, 768, ln.PATH_SCALAR),
])
def test_forward_stores_the_oracle_decisions(dtype, rows, cols, path):
    p, seed, offset = 0.25, 2 ** 36 + 9, 1000 + rows
    inp = synth.make_inputs(rows, cols, dtype, seed=cols)
    bias = synth.make_inputs(1, cols, dtype, seed=3, x=("normal", 0.0, 0.1))["x"][0].cuda()
    d = P.to_device(inp)
    keep = torch.full((ln.dropout_keep_bytes(rows, cols),), 0xAA, dtype=torch.uint8, device="cuda")
    ln.force_path(path)
    a = ln.fwd_bias_dropout(d["x"], bias, d["res"], d["gamma"], d["beta"], EPS, p, seed, offset)
    b = ln.fwd_bias_dropout(d["x"], bias, d["res"], d["gamma"], d["beta"], EPS, p, seed, offset,
                            keep=keep)
    torch.cuda.synchronize()
    got = keep.cpu().numpy().reshape(rows, (cols + 7) // 8)
    np.testing.assert_array_equal(got, oracle_keep_bytes(seed, offset, p, rows, cols))
    for k in range(4):  # storing the bits changes nothing else
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(300, 768), (300, 1001), (8192, 768), (7, 1004)])
def test_backward_from_stored_bits_is_the_generator_backward(dtype, rows, cols):
    if dtype == "bf16" and cols == 1004:
        cols = 1000
    p, seed, offset = 0.1, 5, 17
    inp = synth.make_inputs(rows, cols, dtype, seed=7)
    d = P.to_device(inp)
    bias = torch.zeros(cols, dtype=d["x"].dtype, device="cuda")
    keep = torch.empty(ln.dropout_keep_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    ln.fwd_bias_dropout(d["x"], bias, d["res"], d["gamma"], d["beta"], EPS, p, seed, offset,
                        keep=keep)
    a = ln.dropout_bwd(d["dy"], p, seed, offset)
    b = ln.dropout_bwd(d["dy"], p, keep=keep)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    ref = oracle.dropout_bwd(P.to64(d["dy"]), p, seed, offset, io=dtype)
    P.compare("dx", P.to64(b[0]), ref["dh"], dtype)


def test_stored_bits_path_full_size_gpt2_small():
    """8192 x 768 bf16, p = 0.1: forward storing the bits, backward reading them, against the
    oracle; the workspace is left zero."""
    rows, cols, p, seed, offset = 8192, 768, 0.1, 1234, 0
    inp = synth.make_inputs(rows, cols, "bf16", seed=rows + cols)
    bias = synth.make_inputs(1, cols, "bf16", seed=3, x=("normal", 0.0, 0.1))["x"][0]
    d = P.to_device(inp)
    keep = torch.empty(ln.dropout_keep_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(ln.workspace_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    out, res_out, mean, rstd = ln.fwd_bias_dropout(d["x"], bias.cuda(), d["res"], d["gamma"],
                                                   d["beta"], EPS, p, seed, offset, keep=keep)
    dh, dbias = ln.dropout_bwd(d["dy"], p, keep=keep, workspace=ws)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0
    keepm = oracle.dropout_mask(seed, offset, p, rows, cols).astype(bool)
    np.testing.assert_array_equal(P.to64(res_out)[~keepm], P.to64(inp["res"])[~keepm])
    b = oracle.dropout_bwd(P.to64(d["dy"]), p, seed, offset, io="bf16")
    assert P.compare("dx", P.to64(dh), b["dh"], "bf16")["n_over_stated"] == 0
    terms = keepm * P.to64(d["dy"]) / (1 - p)
    allow = 36.0 * 2.0 ** -24 * np.sqrt((terms ** 2).sum(axis=0))
    P.compare("dbeta", P.to64(dbias), b["dbias"], "bf16", extra=allow)

