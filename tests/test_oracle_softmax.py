"""Pins for the float64 oracle of the fused softmax (CPU only).

Forward: "Accelerating Transformer on GPU (I)", section 4.1 (scale, additive mask, row max,
exp, sum, divide).  Backward: "Accelerating Transformer on GPU (II)", section 3.1
(dx = y (dy - sum dy y), y alone is needed).  The oracle is pinned to things other than
itself: the page's worked exercise (golden fixture), torch's float64 softmax and autograd,
the explicit Jacobian diag(y) - y y^T (the page's own cross-check of the formula), central
finite differences, closed forms and invariants (rows sum to 1, dx sums to 0, shift
invariance, a two-entry row is a logistic), and planted mistakes.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import numpy_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, loc=0.0, scale=1.0):
    return np.random.default_rng(seed).normal(loc, scale, size=shape)


def test_worked_exercise():
    g = json.load(open(os.path.join(GOLDEN, "softmax_backward_worked.json")))
    y = np.array([g["y"]])
    dy = np.array([g["dy"]])
    assert float((dy * y).sum()) == g["s"]
    dx = oracle.softmax_bwd(dy, y)
    np.testing.assert_allclose(dx[0], g["dx"], rtol=0, atol=1e-15)
    assert abs(dx.sum()) < 1e-15


@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
def test_forward_matches_torch_softmax(io):
    rows, cols, scale = 9, 37, 0.125
    x = oracle.round_io(_rand((rows, cols), 1, scale=4.0), io)
    mask = np.where(np.random.default_rng(2).random((3, cols)) < 0.25, -np.inf, 0.0)
    y = oracle.softmax_fwd(x, mask, scale, io=io)
    z = scale * torch.tensor(x) + torch.tensor(np.tile(mask, (3, 1)))
    ref = torch.softmax(z, dim=1).numpy()
    if io == "f64":
        np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-16)
    else:
        np.testing.assert_array_equal(y, oracle.round_io(ref, io))
    assert np.all(y[np.isinf(np.tile(mask, (3, 1)))] == 0.0)


def test_forward_invariants_and_closed_forms():
    x = _rand((6, 50), 3, scale=5.0)
    y = oracle.softmax_fwd(x, None, 0.7)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.softmax_fwd(x + 123.25, None, 1.0),
                               oracle.softmax_fwd(x, None, 1.0), rtol=1e-12)
    # Equal entries: 1 / m.  Two entries: a logistic of the difference.
    np.testing.assert_allclose(oracle.softmax_fwd(np.full((2, 8), 3.5)), 1.0 / 8, rtol=1e-15)
    a, b = 0.3, -1.7
    y2 = oracle.softmax_fwd(np.array([[a, b]]), None, 2.0)
    np.testing.assert_allclose(y2[0, 0], 1.0 / (1.0 + np.exp(-2.0 * (a - b))), rtol=1e-15)
    # Large inputs do not overflow (the row maximum is subtracted first).
    big = oracle.softmax_fwd(np.array([[1000.0, 999.0, 0.0]]))
    assert np.all(np.isfinite(big)) and abs(big.sum() - 1.0) < 1e-15
    # A fully masked row has no softmax: 0 / 0.
    assert np.all(np.isnan(oracle.softmax_fwd(np.zeros((1, 4)), np.full((1, 4), -np.inf))))


@pytest.mark.parametrize("cols", [2, 3, 5, 8])
def test_backward_central_finite_differences(cols):
    rows, h, scale = 3, 1e-6, 0.8
    x = _rand((rows, cols), 20 + cols)
    dy = _rand((rows, cols), 30 + cols)

    def loss(x_):
        return float(np.sum(dy * oracle.softmax_fwd(x_, None, scale)))

    y = oracle.softmax_fwd(x, None, scale)
    dx = oracle.softmax_bwd(dy, y, scale)
    for i in range(rows):
        for j in range(cols):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            num = (loss(xp) - loss(xm)) / (2 * h)
            assert abs(num - dx[i, j]) <= 1e-8 * max(1.0, abs(num))


def test_backward_matches_autograd_and_the_jacobian():
    rows, cols, scale = 4, 29, 0.5
    x = _rand((rows, cols), 40, scale=3.0)
    dy = _rand((rows, cols), 41)
    mask = np.where(np.random.default_rng(42).random((1, cols)) < 0.2, -np.inf, 0.0)
    xt = torch.tensor(x, requires_grad=True)
    yt = torch.softmax(scale * xt + torch.tensor(mask), dim=1)
    (yt * torch.tensor(dy)).sum().backward()
    y = oracle.softmax_fwd(x, mask, scale)
    dx = oracle.softmax_bwd(dy, y, scale)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-12, atol=1e-14)
    for r in range(rows):  # the explicit Jacobian diag(y) - y y^T times dy
        J = np.diag(y[r]) - np.outer(y[r], y[r])
        np.testing.assert_allclose(dx[r], scale * J @ dy[r], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dx.sum(axis=1), 0.0, atol=1e-14)


@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
def test_c_oracle_matches_numpy_twin(io):
    rows, cols = 10, 300
    x = oracle.round_io(_rand((rows, cols), 50, scale=3.0), io)
    mask = oracle.round_io(np.where(np.random.default_rng(51).random((5, cols)) < 0.1, -np.inf, 0.0), io)
    dy = oracle.round_io(_rand((rows, cols), 52), io)
    a = oracle.softmax_fwd(x, mask, 0.25, io=io)
    b = numpy_ref.softmax_fwd(x, mask, 0.25, io=io)
    # Summation orders differ (sequential in C, pairwise in NumPy): a few float64 ulps, then
    # at most one step of the I/O rounding.
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(b), 1e-300))) - {"f64": 40, "f32": 23, "bf16": 7}[io])
    assert np.all(np.abs(a - b) <= ulp)
    ga = oracle.softmax_bwd(dy, a, 0.25, io=io)
    gb = numpy_ref.softmax_bwd(dy, a, 0.25, io=io)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(gb), 1e-300))) - {"f64": 40, "f32": 23, "bf16": 7}[io])
    assert np.all(np.abs(ga - gb) <= ulp)


def _mutant(kind):
    def fwd(x):
        if kind == "no_max_shift":
            e = np.exp(x)
        elif kind == "max_not_subtracted_in_sum":
            e = np.exp(x - x.max(axis=1, keepdims=True))
            return e / np.exp(x).sum(axis=1, keepdims=True)
        else:
            raise ValueError(kind)
        return e / e.sum(axis=1, keepdims=True)
    return fwd


@pytest.mark.parametrize("kind", ["no_max_shift", "max_not_subtracted_in_sum"])
def test_pins_catch_planted_forward_mistakes(kind):
    x = np.array([[1000.0, 999.0, 0.0], [0.5, 1.5, -2.0]])
    with np.errstate(all="ignore"):
        bad = _mutant(kind)(x)
    ref = torch.softmax(torch.tensor(x), dim=1).numpy()
    assert not np.allclose(bad, ref, equal_nan=False)
    np.testing.assert_allclose(numpy_ref.softmax_fwd(x), ref, rtol=1e-14)


@pytest.mark.parametrize("kind", ["sign", "no_y_factor", "no_scale"])
def test_pins_catch_planted_backward_mistakes(kind):
    scale = 0.5
    x = _rand((3, 6), 60)
    dy = _rand((3, 6), 61)
    y = numpy_ref.softmax_fwd(x, None, scale)
    s = (dy * y).sum(axis=1, keepdims=True)
    bad = {"sign": scale * y * (dy + s), "no_y_factor": scale * (dy - s),
           "no_scale": y * (dy - s)}[kind]
    xt = torch.tensor(x, requires_grad=True)
    (torch.softmax(scale * xt, dim=1) * torch.tensor(dy)).sum().backward()
    assert np.max(np.abs(bad - xt.grad.numpy())) > 1e-3
    np.testing.assert_allclose(numpy_ref.softmax_bwd(dy, y, scale), xt.grad.numpy(), rtol=1e-12,
                               atol=1e-15)
