"""Pins for the float64 oracle of the bias + dropout + residual prologue of the LayerNorm
forward ("Accelerating Transformer on GPU (I)", section 2.3) and its backward (CPU only).

The pages fix no random-number generator for the dropout mask; the oracle takes the
counter-based Philox-4x32-10 of Salmon, Moraes, Dror and Shaw ("Parallel Random Numbers: As
Easy as 1, 2, 3", SC 2011), written from that paper's definition.  It is pinned to the
generator's published known-answer vectors, to an independent NumPy restatement, to the
statistics of the mask, to closed forms (p = 0 is the plain fused residual LayerNorm; dropped
elements contribute nothing), and to torch float64 autograd of the composed function with
the same mask.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import numpy_ref

# Known-answer vectors published with the Random123 implementation of Philox-4x32-10
# (counter, key) -> output.
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", KAT)
def test_philox_known_answers(ctr, key, out):
    assert tuple(oracle.philox4x32(ctr, key)) == out
    w = numpy_ref.philox4x32(*[np.array([c], dtype=np.uint64) for c in ctr], *key)
    assert tuple(int(v[0]) for v in w) == out


def test_mask_matches_numpy_twin_and_its_statistics():
    for seed, offset, p in ((1, 0, 0.1), (2**40 + 7, 2**33 + 5, 0.5), (99, 3, 0.0)):
        a = oracle.dropout_mask(seed, offset, p, 200, 333)
        b = numpy_ref.dropout_mask(seed, offset, p, 200, 333)
        assert np.array_equal(a, b)
        n = a.size
        kept = a.mean()
        assert abs(kept - (1 - p)) <= 5 * np.sqrt(p * (1 - p) / n) + 1e-12
    # Different offsets give different masks; the same arguments give the same mask.
    assert not np.array_equal(oracle.dropout_mask(1, 0, 0.5, 64, 64),
                              oracle.dropout_mask(1, 1, 0.5, 64, 64))
    assert np.array_equal(oracle.dropout_mask(5, 9, 0.3, 64, 64),
                          oracle.dropout_mask(5, 9, 0.3, 64, 64))


def _inputs(rows, cols, seed):
    rng = np.random.default_rng(seed)
    return (rng.normal(0, 1, (rows, cols)), rng.normal(0, 0.1, cols), rng.normal(0, 1, (rows, cols)),
            rng.normal(1, 0.1, cols), rng.normal(0, 0.1, cols))


def test_zero_probability_is_the_fused_residual_layernorm():
    h, b, r, g, be = _inputs(6, 40, 1)
    a = oracle.bdr_ln_fwd(h, b, r, g, be, 1e-5, 0.0, 3, 4)
    ref = oracle.ln_fwd(h + b[None, :], r, g, be, 1e-5)
    for k in ("out", "res_out", "mean", "rstd"):
        np.testing.assert_allclose(a[k], ref[k], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
def test_forward_matches_numpy_twin_and_drops(io):
    h, b, r, g, be = _inputs(9, 64, 2)
    h, r = oracle.round_io(h, io), oracle.round_io(r, io)
    p = 0.25
    a = oracle.bdr_ln_fwd(h, b, r, g, be, 1e-5, p, 11, 22, io=io)
    n = numpy_ref.bdr_ln_fwd(h, b, r, g, be, 1e-5, p, 11, 22, io=io)
    np.testing.assert_array_equal(a["res_out"], n["res_out"])
    keep = oracle.dropout_mask(11, 22, p, 9, 64)
    np.testing.assert_array_equal(a["res_out"][keep == 0], r[keep == 0])
    np.testing.assert_allclose(a["mean"], n["mean"], rtol=1e-13, atol=1e-15)


def test_backward_matches_autograd_with_the_same_mask():
    rows, cols, p, eps = 5, 24, 0.3, 1e-5
    h, b, r, g, be = _inputs(rows, cols, 3)
    dy = np.random.default_rng(4).normal(0, 1, (rows, cols))
    keep = torch.tensor(oracle.dropout_mask(7, 8, p, rows, cols), dtype=torch.float64)
    ht = torch.tensor(h, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    rt = torch.tensor(r, requires_grad=True)
    s = rt + keep * (ht + bt) / (1 - p)
    y = torch.nn.functional.layer_norm(s, (cols,), torch.tensor(g), torch.tensor(be), eps)
    (y * torch.tensor(dy)).sum().backward()
    f = oracle.bdr_ln_fwd(h, b, r, g, be, eps, p, 7, 8)
    np.testing.assert_allclose(f["out"], y.detach().numpy(), rtol=1e-12, atol=1e-13)
    ds = oracle.ln_bwd(dy, f["res_out"], g, f["mean"], f["rstd"])["dx"]
    np.testing.assert_allclose(ds, rt.grad.numpy(), rtol=1e-11, atol=1e-12)
    back = oracle.dropout_bwd(ds, p, 7, 8)
    np.testing.assert_allclose(back["dh"], ht.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(back["dbias"], bt.grad.numpy(), rtol=1e-11, atol=1e-12)
    nb = numpy_ref.dropout_bwd(ds, p, 7, 8)
    np.testing.assert_allclose(back["dh"], nb["dh"], rtol=1e-15)
    np.testing.assert_allclose(back["dbias"], nb["dbias"], rtol=1e-13, atol=1e-15)


def test_planted_mistakes_are_caught():
    """Scaling by (1 - p) instead of dividing, or reusing one word for all four elements of a
    counter, changes the results the pins above check."""
    rows, cols, p = 4, 16, 0.4
    keep = oracle.dropout_mask(1, 2, p, rows, cols)
    i = np.arange(rows * cols, dtype=np.uint64)
    blk = i >> np.uint64(2)
    w = numpy_ref.philox4x32(blk & np.uint64(0xFFFFFFFF), blk >> np.uint64(32),
                             np.full_like(blk, 2), np.zeros_like(blk), 1, 0)
    one_word = (w[0] >= np.uint64(int(p * 2 ** 32))).astype(np.uint8).reshape(rows, cols)
    assert not np.array_equal(one_word, keep)
    ds = np.ones((rows, cols))
    good = oracle.dropout_bwd(ds, p, 1, 2)["dh"]
    assert not np.allclose(good, keep * ds * (1 - p))
