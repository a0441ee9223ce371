"""Parity of the fused softmax kernels (called through the C ABI) with the float64 oracle:
"Accelerating Transformer on GPU (I)", section 4.1 (forward: scale, additive mask, max,
exp, sum, divide) and "... (II)", section 3.1 (backward from y alone).  Every kernel family,
ragged and unaligned rows, masks that repeat every L rows (a causal attention mask), fully
masked rows, large scores, and the pages' attention shapes at full size on every row.
Tolerances are those of ``lnparity`` (fp32 2e-5, bf16 2 ulps)."""
import numpy as np
import pytest
import torch

import layernorm_ln_fwd_gb300 as ln
import lnparity as P
import oracle
from layernorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _auto_path():
    ln.force_path(ln.PATH_AUTO)
    yield
    ln.force_path(ln.PATH_AUTO)


def causal_mask(L, cols, dtype):
    m = torch.zeros(L, cols)
    q = torch.arange(L)[:, None]
    k = torch.arange(cols)[None, :]
    m[k > q * cols // L] = float("-inf")
    return m.to(synth.torch_dtype(dtype))


def inputs(rows, cols, dtype, seed, spread=3.0):
    inp = synth.make_inputs(rows, cols, dtype, seed=seed, x=("normal", 0.0, spread))
    return inp["x"], inp["dy"]


def check(x, dy, mask, scale, dtype, aliased=False):
    io = dtype
    d_x, d_dy = x.cuda(), dy.cuda()
    d_mask = mask.cuda() if mask is not None else None
    y = ln.softmax_fwd(d_x, d_mask, scale)
    dx = ln.softmax_bwd(d_dy, y, scale, dx=d_dy if aliased else None)
    torch.cuda.synchronize()
    ref_y = oracle.softmax_fwd(P.to64(x), None if mask is None else P.to64(mask), scale, io=io)
    ref_dx = oracle.softmax_bwd(P.to64(dy), P.to64(y), scale, io=io)
    gy, gdx = P.to64(y), P.to64(dx)
    nan = np.isnan(ref_y)
    assert np.array_equal(np.isnan(gy), nan)
    infos = [P.compare("y", gy[~nan], ref_y[~nan], io)]
    nan_dx = np.isnan(ref_dx)
    assert np.array_equal(np.isnan(gdx), nan_dx)
    infos.append(P.compare("dx", gdx[~nan_dx], ref_dx[~nan_dx], io))
    return infos


COLS = [1, 3, 8, 32, 33, 128, 256, 512, 1000, 1001, 1024, 2048, 2056, 4096, 8192, 16384]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", [1, 300])
def test_shapes_against_oracle(dtype, rows, cols):
    x, dy = inputs(rows, cols, dtype, seed=rows + cols)
    check(x, dy, None, 1.0, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", [ln.PATH_WARP, ln.PATH_BLOCK, ln.PATH_SCALAR])
@pytest.mark.parametrize("rows,cols", [(5, 64), (37, 512), (64, 1024), (19, 1000), (9, 4104)])
def test_every_kernel_family_with_a_causal_mask(dtype, path, rows, cols):
    if dtype == "bf16" and cols == 1000:
        cols = 1000 - 8
    ln.force_path(path)
    x, dy = inputs(rows, cols, dtype, seed=7 + path)
    check(x, dy, causal_mask(min(rows, 16), cols, dtype), 0.125, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", [ln.PATH_AUTO, ln.PATH_BLOCK, ln.PATH_SCALAR])
def test_fully_masked_rows_and_large_scores(dtype, path):
    """Rows whose mask removes every entry give NaN (0/0, as the definition does) without
    touching the other rows; scores of +-1000 do not overflow (the row max is taken first)."""
    ln.force_path(path)
    rows, cols = 24, 256
    x, dy = inputs(rows, cols, dtype, seed=5, spread=300.0)
    mask = torch.zeros(4, cols)
    mask[1] = float("-inf")          # every 4th row from row 1: fully masked
    mask[2, : cols // 2] = float("-inf")
    check(x, dy, mask.to(synth.torch_dtype(dtype)), 1.0, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gradient_may_overwrite_dy(dtype):
    x, dy = inputs(50, 768, dtype, seed=9)
    check(x, dy, None, 0.5, dtype, aliased=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unaligned_pointers_take_the_scalar_kernel(dtype):
    rows, cols = 17, 512
    x, dy = inputs(rows, cols, dtype, seed=11)
    td = synth.torch_dtype(dtype)

    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=td, device="cuda")
        v = buf[1:].view(t.shape)
        v.copy_(t.cuda())
        return v

    sx, sdy = shifted(x), shifted(dy)
    y = ln.softmax_fwd(sx, None, 1.0, y=shifted(x))
    dx = ln.softmax_bwd(sdy, y, 1.0, dx=shifted(x))
    torch.cuda.synchronize()
    P.compare("y", P.to64(y), oracle.softmax_fwd(P.to64(x), None, 1.0, io=dtype), dtype)
    P.compare("dx", P.to64(dx), oracle.softmax_bwd(P.to64(dy), P.to64(y), 1.0, io=dtype), dtype)


@pytest.mark.parametrize("dtype,batch,heads,L", [("bf16", 8, 16, 512), ("bf16", 2, 16, 256),
                                                 ("f32", 2, 16, 256)])
def test_attention_shapes_full_size(dtype, batch, heads, L):
    """The attention scores the pages size their estimates on (batch x heads x L x L: 8 x 16
    x 512 x 512, "... (II)", section 3.2; 2 x 16 x 256 x 256, "... (I)", section 4.1), with a
    causal mask and the 1/sqrt(64) scale, every row compared; the backward is bitwise
    repeatable."""
    rows = batch * heads * L
    x, dy = inputs(rows, L, dtype, seed=0)
    infos = check(x, dy, causal_mask(L, L, dtype), 0.125, dtype)
    assert all(i["n_over_stated"] == 0 for i in infos)
    d_y = ln.softmax_fwd(x.cuda(), causal_mask(L, L, dtype).cuda(), 0.125)
    a = ln.softmax_bwd(dy.cuda(), d_y, 0.125)
    b = ln.softmax_bwd(dy.cuda(), d_y, 0.125)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_launch_count():
    x = torch.randn(64, 512, device="cuda")
    y = ln.softmax_fwd(x)
    assert ln.last_launch_count() == 1
    ln.softmax_bwd(x, y)
    assert ln.last_launch_count() == 1
