"""Pins for the float64 oracle of the fused residual-add + RMSNorm (CPU only).

The page ("GPU Performance from First Principles", section 6.1 and exercise 4) names the
operation -- read x and the residual, write the new residual stream and the normalised
result -- without printing a formula; the oracle takes the usual RMSNorm (no mean
subtracted, no shift, eps inside the square root, a per-column gain).  It is pinned here to
things other than itself: torch's own float64 rms_norm and its autograd, central finite
differences, closed forms (constant rows, one column, the scale invariance at eps = 0, the
projection identity sum_j dx_j s_j = r^3 eps sum_j g_j s_j), the NumPy twin, and the page's
count of vector passes.  ``test_pins_catch_planted_mistakes`` plants plausible slips in a
copy of the NumPy twin and shows that the pins catch them.
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


def _torch_rms(s, gamma, eps):
    return torch.nn.functional.rms_norm(s, (s.shape[-1],), gamma, eps)


@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
def test_forward_matches_torch_rms_norm(io):
    rows, cols, eps = 7, 33, 1e-5
    x = oracle.round_io(_rand((rows, cols), 1), io)
    res = oracle.round_io(_rand((rows, cols), 2), io)
    gamma = oracle.round_io(_rand(cols, 3, 1.0, 0.1), io)
    r = oracle.rms_fwd(x, res, gamma, eps, io=io)
    np.testing.assert_array_equal(r["res_out"], oracle.round_io(x + res, io))
    s64 = torch.tensor(r["res_out"], dtype=torch.float64)
    ref = _torch_rms(s64, torch.tensor(gamma), eps).numpy()
    if io == "f64":
        np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-13)
    else:
        np.testing.assert_array_equal(r["out"], oracle.round_io(ref, io))
    ms = (r["res_out"] ** 2).mean(axis=1)
    np.testing.assert_allclose(r["rrms"], 1.0 / np.sqrt(ms + eps), rtol=1e-14)


def test_forward_closed_forms():
    eps = 1e-5
    gamma = np.array([1.5, -2.0, 0.25])
    # A constant row c: r = 1/sqrt(c^2 + eps); with eps = 0 the output is gamma * sign(c).
    r = oracle.rms_fwd(np.array([[7.25] * 3, [-4.0] * 3]), None, gamma, 0.0)
    np.testing.assert_allclose(r["out"], [gamma, -gamma], rtol=1e-15)
    r = oracle.rms_fwd(np.array([[3.0] * 3]), None, gamma, eps)
    np.testing.assert_allclose(r["rrms"], [1.0 / np.sqrt(9.0 + eps)], rtol=1e-15)
    # One column: out = gamma * s / sqrt(s^2 + eps), dx = r * g * eps / (s^2 + eps).
    s = np.array([[3.0], [-0.5]])
    r1 = oracle.rms_fwd(s, None, np.array([2.0]), eps)
    np.testing.assert_allclose(r1["out"][:, 0], 2.0 * s[:, 0] / np.sqrt(s[:, 0] ** 2 + eps),
                               rtol=1e-15)
    dy = np.array([[1.0], [-2.0]])
    b1 = oracle.rms_bwd(dy, s, np.array([2.0]), r1["rrms"])
    rr = r1["rrms"]
    np.testing.assert_allclose(b1["dx"][:, 0], rr * 2.0 * dy[:, 0] * eps * rr ** 2, rtol=1e-9)
    # gamma = 1: every output row has mean square ms / (ms + eps).
    x = _rand((16, 257), 5, scale=0.003)  # small ms makes eps visible
    r2 = oracle.rms_fwd(x, None, np.ones(257), eps)
    ms = (x ** 2).mean(axis=1)
    np.testing.assert_allclose((r2["out"] ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12)
    assert np.all(ms / (ms + eps) < 0.9)


def test_scale_invariance_at_zero_eps():
    x = _rand((4, 9), 7)
    gamma = _rand(9, 8, 1.0, 0.1)
    a = oracle.rms_fwd(x, None, gamma, 0.0)["out"]
    b = oracle.rms_fwd(x * 37.5, None, gamma, 0.0)["out"]
    np.testing.assert_allclose(a, b, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("cols", [1, 2, 3, 5, 8])
def test_backward_central_finite_differences(cols):
    rows, eps, h = 3, 1e-5, 1e-6
    x = _rand((rows, cols), 20 + cols)
    res = _rand((rows, cols), 30 + cols)
    dy = _rand((rows, cols), 40 + cols)
    gamma = _rand(cols, 50 + cols, 1.0, 0.1)

    def loss(x_, res_, g_):
        return float(np.sum(dy * oracle.rms_fwd(x_, res_, g_, eps)["out"]))

    f = oracle.rms_fwd(x, res, gamma, eps)
    b = oracle.rms_bwd(dy, f["res_out"], gamma, f["rrms"])
    for (i, j) in [(r, c) for r in range(rows) for c in range(cols)]:
        for which in ("x", "res"):
            xp, xm = x.copy(), x.copy()
            rp, rm = res.copy(), res.copy()
            (xp if which == "x" else rp)[i, j] += h
            (xm if which == "x" else rm)[i, j] -= h
            num = (loss(xp, rp, gamma) - loss(xm, rm, gamma)) / (2 * h)
            assert abs(num - b["dx"][i, j]) <= 1e-7 * max(1.0, abs(num)), (which, i, j)
    for j in range(cols):
        gp, gm = gamma.copy(), gamma.copy()
        gp[j] += h
        gm[j] -= h
        num = (loss(x, res, gp) - loss(x, res, gm)) / (2 * h)
        assert abs(num - b["dgamma"][j]) <= 1e-7 * max(1.0, abs(num))


@pytest.mark.parametrize("rows,cols", [(6, 17), (3, 256)])
def test_backward_matches_torch_autograd(rows, cols):
    eps = 1e-5
    x = _rand((rows, cols), 60)
    res = _rand((rows, cols), 61)
    dy = _rand((rows, cols), 62)
    gamma = _rand(cols, 63, 1.0, 0.1)
    xt = torch.tensor(x, requires_grad=True)
    rt = torch.tensor(res, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    y = _torch_rms(xt + rt, gt, eps)
    (y * torch.tensor(dy)).sum().backward()
    f = oracle.rms_fwd(x, res, gamma, eps)
    b = oracle.rms_bwd(dy, f["res_out"], gamma, f["rrms"])
    np.testing.assert_allclose(b["dx"], xt.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dx"], rt.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["dgamma"], gt.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_backward_projection_identity():
    """sum_j dx_j s_j = r^3 eps sum_j g_j s_j per row (so 0 at eps = 0: the output does not
    change when s is scaled, and the gradient is orthogonal to s)."""
    rows, cols = 5, 40
    s = _rand((rows, cols), 70)
    dy = _rand((rows, cols), 71)
    gamma = _rand(cols, 72, 1.0, 0.1)
    for eps in (0.0, 1e-5, 0.3):
        f = oracle.rms_fwd(s, None, gamma, eps)
        b = oracle.rms_bwd(dy, s, gamma, f["rrms"])
        lhs = (b["dx"] * s).sum(axis=1)
        rhs = f["rrms"] ** 3 * eps * (gamma[None, :] * dy * s).sum(axis=1)
        np.testing.assert_allclose(lhs, rhs, rtol=1e-9, atol=1e-12)


def test_column_gradient_is_a_row_ordered_sum():
    s = _rand((40, 6), 80)
    dy = _rand((40, 6), 81)
    f = oracle.rms_fwd(s, None, np.ones(6), 1e-5)
    b = oracle.rms_bwd(dy, s, np.ones(6), f["rrms"])
    ref = np.zeros(6)
    for r in range(40):
        ref += dy[r] * (s[r] * f["rrms"][r])
    np.testing.assert_array_equal(b["dgamma"], ref)


@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(9, 31), (4, 1000)])
def test_c_oracle_matches_numpy_twin(io, rows, cols):
    eps = 1e-5
    x = oracle.round_io(_rand((rows, cols), 90), io)
    res = oracle.round_io(_rand((rows, cols), 91), io)
    dy = oracle.round_io(_rand((rows, cols), 92), io)
    gamma = oracle.round_io(_rand(cols, 93, 1.0, 0.1), io)
    a = oracle.rms_fwd(x, res, gamma, eps, io=io)
    b = numpy_ref.rms_fwd(x, res, gamma, eps, io=io)
    np.testing.assert_array_equal(a["res_out"], b["res_out"])
    np.testing.assert_allclose(a["rrms"], b["rrms"], rtol=1e-14)
    np.testing.assert_allclose(a["out"], b["out"], rtol=2e-16 if io == "f64" else 0,
                               atol=1e-15 if io == "f64" else 2.0 ** -7 * np.abs(b["out"]).max())
    ga = oracle.rms_bwd(dy, a["res_out"], gamma, a["rrms"], io=io)
    gb = numpy_ref.rms_bwd(dy, b["res_out"], gamma, b["rrms"], io=io)
    for k in ("dx", "dgamma"):
        if io == "f64":
            np.testing.assert_allclose(ga[k], gb[k], rtol=1e-12, atol=1e-13)
        else:  # the same value before rounding: differences only by one rounding step
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(gb[k]), 1e-30))) -
                          (23 if io == "f32" else 7))
            assert np.all(np.abs(ga[k] - gb[k]) <= ulp)


def test_fused_pass_count_matches_the_page():
    """The page's count of vector passes of the residual add + RMSNorm, and the algorithmic
    bytes the benchmark charges the fused forward: reads of x and the residual, writes of the
    new residual stream and the normalised result (plus gamma and the per-row statistic)."""
    g = json.load(open(os.path.join(GOLDEN, "fused_add_rmsnorm_passes.json")))
    unfused = g["unfused_reads"] + g["unfused_writes"]
    fused = g["fused_reads"] + g["fused_writes"]
    assert (unfused - fused) / unfused == g["saving"]
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    R, C, s = 1000, 512, 2
    assert bench.rms_fwd_bytes(R, C, s) == fused * R * C * s + C * s + 4 * R


def _mutant_fwd(kind):
    def fwd(x, gamma, eps):
        x = np.asarray(x, dtype=np.float64)
        if kind == "mean_subtracted":
            x = x - x.mean(axis=1, keepdims=True)
            ms = (x * x).mean(axis=1)
        elif kind == "unbiased_divisor":
            ms = (x * x).sum(axis=1) / (x.shape[1] - 1)
        elif kind == "eps_outside":
            return gamma[None, :] * x / (np.sqrt((x * x).mean(axis=1)) + eps)[:, None]
        else:
            raise ValueError(kind)
        return gamma[None, :] * x / np.sqrt(ms + eps)[:, None]
    return fwd


def _mutant_bwd(kind):
    def bwd(dy, s, gamma, rrms):
        m = dy.shape[1]
        shat = s * rrms[:, None]
        g = gamma[None, :] * dy
        sgs = (g * shat).sum(axis=1, keepdims=True)
        if kind == "dropped_term":
            return rrms[:, None] * g
        if kind == "wrong_sign":
            return rrms[:, None] * (g + shat * sgs / m)
        if kind == "layernorm_mean_term":
            return rrms[:, None] * (g - (g.sum(axis=1, keepdims=True) + shat * sgs) / m)
        raise ValueError(kind)
    return bwd


@pytest.mark.parametrize("kind", ["mean_subtracted", "unbiased_divisor", "eps_outside"])
def test_pins_catch_planted_forward_mistakes(kind):
    x = _rand((3, 6), 101, loc=0.05, scale=0.01)  # a visible mean and a small, eps-sized ms
    gamma = _rand(6, 102, 1.0, 0.1)
    eps = 1e-3
    bad = _mutant_fwd(kind)(x, gamma, eps)
    ref = _torch_rms(torch.tensor(x), torch.tensor(gamma), eps).numpy()
    assert np.max(np.abs(bad - ref)) > 1e-4
    good = numpy_ref.rms_fwd(x, None, gamma, eps)["out"]
    np.testing.assert_allclose(good, ref, rtol=1e-13)


@pytest.mark.parametrize("kind", ["dropped_term", "wrong_sign", "layernorm_mean_term"])
def test_pins_catch_planted_backward_mistakes(kind):
    rows, cols, eps = 3, 5, 1e-5
    x = _rand((rows, cols), 111, loc=0.3)
    dy = _rand((rows, cols), 112)
    gamma = _rand(cols, 113, 1.0, 0.1)
    f = numpy_ref.rms_fwd(x, None, gamma, eps)
    bad = _mutant_bwd(kind)(dy, f["res_out"], gamma, f["rrms"])
    xt = torch.tensor(x, requires_grad=True)
    (_torch_rms(xt, torch.tensor(gamma), eps) * torch.tensor(dy)).sum().backward()
    assert np.max(np.abs(bad - xt.grad.numpy())) > 1e-3
    good = numpy_ref.rms_bwd(dy, f["res_out"], gamma, f["rrms"])["dx"]
    np.testing.assert_allclose(good, xt.grad.numpy(), rtol=1e-12, atol=1e-13)
