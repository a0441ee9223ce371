"""Pins for the float64 oracle (CPU only).

The oracle is checked against things other than itself: numbers the pages print, closed
forms, invariants, finite differences, and torch's own float64 layer_norm and autograd.
Each check is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign,
a transposed operand, the unbiased variance, eps outside the square root, a wrong rounding)
fails at least one of them; ``test_pins_catch_planted_mistakes`` plants such slips in a copy
of the NumPy twin and shows that they are caught.
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


def _ln_params(cols, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(1.0, 0.1, cols), rng.normal(0.0, 0.1, cols)


# ----------------------------------------------------------------------------------------
# Worked example printed on the pages
# ----------------------------------------------------------------------------------------
def test_worked_example_two_values():
    g = json.load(open(os.path.join(GOLDEN, "two_values_1000_1001.json")))
    row = np.array([g["row"]])
    # The printed intermediate values are consistent with each other.
    assert np.mean(row) == g["E_x"]
    assert np.mean(row) ** 2 == g["E_x_squared"]
    assert np.mean(row ** 2) == g["E_x2"]
    # The oracle reproduces the printed mean and variance (eps = 0: rstd = 1/sqrt(var)).
    r = oracle.ln_fwd(row, None, np.ones(2), np.zeros(2), 0.0, io="f64")
    assert r["mean"][0] == g["E_x"]
    assert r["rstd"][0] == 1.0 / np.sqrt(g["var"])
    np.testing.assert_array_equal(r["out"], [[-1.0, 1.0]])
    np.testing.assert_array_equal(r["res_out"], row)


# ----------------------------------------------------------------------------------------
# Forward pins
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
def test_forward_matches_torch_layer_norm(io):
    rows, cols = 7, 33
    x = oracle.round_io(_rand((rows, cols), 1), io)
    res = oracle.round_io(_rand((rows, cols), 2), io)
    gamma, beta = (oracle.round_io(p, io) for p in _ln_params(cols, 3))
    eps = 1e-5
    r = oracle.ln_fwd(x, res, gamma, beta, eps, io=io)
    # Residual sum, rounded to the stored precision (checked against torch's own casts).
    tdt = {"f64": torch.float64, "f32": torch.float32, "bf16": torch.bfloat16}[io]
    s_t = (torch.tensor(x).to(tdt).float() + torch.tensor(res).to(tdt).float()).to(tdt) \
        if io != "f64" else torch.tensor(x) + torch.tensor(res)
    np.testing.assert_array_equal(r["res_out"], s_t.double().numpy())
    # Normalised output against torch's float64 layer_norm of the stored residual.
    s64 = torch.tensor(r["res_out"], dtype=torch.float64)
    ref = torch.nn.functional.layer_norm(s64, (cols,), torch.tensor(gamma), torch.tensor(beta), eps)
    if io == "f64":
        np.testing.assert_allclose(r["out"], ref.numpy(), rtol=0, atol=1e-13)
    else:
        # Same value before rounding; the rounding is pinned separately.
        np.testing.assert_array_equal(r["out"], oracle.round_io(ref.numpy(), io))
    np.testing.assert_allclose(r["mean"], s64.mean(dim=1).numpy(), rtol=1e-14, atol=1e-15)
    var = s64.var(dim=1, unbiased=False).numpy()
    np.testing.assert_allclose(r["rstd"], 1.0 / np.sqrt(var + eps), rtol=1e-14)


def test_forward_normalised_rows_have_mean_zero_and_known_variance():
    """With gamma = 1, beta = 0 each output row has mean 0 and variance var/(var + eps)."""
    rows, cols = 16, 257
    x = _rand((rows, cols), 5, loc=3.0, scale=0.01)  # small var makes eps visible
    eps = 1e-5
    r = oracle.ln_fwd(x, None, np.ones(cols), np.zeros(cols), eps, io="f64")
    out = r["out"]
    var = x.var(axis=1)
    assert np.max(np.abs(out.mean(axis=1))) < 1e-12
    np.testing.assert_allclose(out.var(axis=1), var / (var + eps), rtol=1e-12)
    assert np.all(var / (var + eps) < 0.95)  # eps is not negligible in this case


def test_forward_constant_row_and_single_column():
    eps = 1e-5
    gamma, beta = np.array([1.5, -2.0, 0.25]), np.array([0.1, -0.2, 0.3])
    r = oracle.ln_fwd(np.full((2, 3), 7.25), None, gamma, beta, eps, io="f64")
    np.testing.assert_array_equal(r["out"], np.stack([beta, beta]))
    np.testing.assert_allclose(r["rstd"], 1.0 / np.sqrt(eps), rtol=1e-15)
    np.testing.assert_array_equal(r["mean"], [7.25, 7.25])
    r1 = oracle.ln_fwd(np.array([[3.0], [-4.0]]), None, np.array([2.0]), np.array([0.5]), eps,
                       io="f64")
    np.testing.assert_array_equal(r1["out"], [[0.5], [0.5]])
    b1 = oracle.ln_bwd(np.array([[1.0], [-2.0]]), np.array([[3.0], [-4.0]]), np.array([2.0]),
                       r1["mean"], r1["rstd"], io="f64")
    np.testing.assert_array_equal(b1["dx"], [[0.0], [0.0]])


def _welford_chan(row, chunk=7):
    """Variance by Welford per chunk and the Chan pairwise merge printed in
    "Accelerating Transformer on GPU (I)", section 4.2 (an independent algorithm)."""
    n, mu, m2 = 0, 0.0, 0.0
    for start in range(0, len(row), chunk):
        part = row[start:start + chunk]
        nb, mub, m2b = 0, 0.0, 0.0
        for v in part:
            nb += 1
            d = v - mub
            mub += d / nb
            m2b += d * (v - mub)
        if n == 0:
            n, mu, m2 = nb, mub, m2b
            continue
        nn = n + nb
        delta = mub - mu
        mu = mu + delta * nb / nn
        m2 = m2 + m2b + delta * delta * n * nb / nn
        n = nn
    return mu, m2 / n


def test_cancellation_large_mean():
    """Rows ~ N(1e4, 1): the one-pass fp32 E[x^2]-E[x]^2 gives var <= 0 for some rows
    ("Accelerating Transformer on GPU (I)", section 4.2) while the oracle's two-pass float64
    variance agrees with a Welford/Chan merge."""
    rows, cols = 64, 256
    x = _rand((rows, cols), 11, loc=1e4, scale=1.0).astype(np.float32).astype(np.float64)
    x32 = x.astype(np.float32)
    naive = np.mean(x32 * x32, axis=1, dtype=np.float32) - np.mean(x32, axis=1, dtype=np.float32) ** 2
    assert np.any(naive <= 0.0)
    r = oracle.ln_fwd(x, None, np.ones(cols), np.zeros(cols), 0.0, io="f64")
    for i in range(rows):
        mu, var = _welford_chan(x[i])
        assert abs(r["mean"][i] - mu) <= 1e-12 * abs(mu)
        assert abs(1.0 / r["rstd"][i] ** 2 - var) <= 1e-9 * var
    assert np.all(1.0 / r["rstd"] ** 2 > 0.5)


# ----------------------------------------------------------------------------------------
# Backward pins
# ----------------------------------------------------------------------------------------
def _loss_and_fwd(x, res, gamma, beta, dy, eps):
    r = oracle.ln_fwd(x, res, gamma, beta, eps, io="f64")
    return float(np.sum(dy * r["out"])), r


@pytest.mark.parametrize("cols", [2, 3, 5, 8])
def test_backward_central_finite_differences(cols):
    rows, eps, h = 3, 1e-5, 1e-6
    x = _rand((rows, cols), 20 + cols)
    res = _rand((rows, cols), 30 + cols)
    dy = _rand((rows, cols), 40 + cols)
    gamma, beta = _ln_params(cols, 50 + cols)
    _, r = _loss_and_fwd(x, res, gamma, beta, dy, eps)
    b = oracle.ln_bwd(dy, r["res_out"], gamma, r["mean"], r["rstd"], io="f64")

    def fd(arr_name, idx):
        args = {"x": x, "res": res, "gamma": gamma, "beta": beta}
        plus = {k: v.copy() for k, v in args.items()}
        minus = {k: v.copy() for k, v in args.items()}
        plus[arr_name][idx] += h
        minus[arr_name][idx] -= h
        lp, _ = _loss_and_fwd(plus["x"], plus["res"], plus["gamma"], plus["beta"], dy, eps)
        lm, _ = _loss_and_fwd(minus["x"], minus["res"], minus["gamma"], minus["beta"], dy, eps)
        return (lp - lm) / (2 * h)

    scale = max(1.0, np.max(np.abs(b["dx"])))
    for i in range(rows):
        for j in range(cols):
            # dx is the gradient of the residual sum, hence of both x and res.
            assert abs(fd("x", (i, j)) - b["dx"][i, j]) <= 1e-7 * scale
            assert abs(fd("res", (i, j)) - b["dx"][i, j]) <= 1e-7 * scale
    for j in range(cols):
        assert abs(fd("gamma", (j,)) - b["dgamma"][j]) <= 1e-7 * max(1, abs(b["dgamma"][j]))
        assert abs(fd("beta", (j,)) - b["dbeta"][j]) <= 1e-7 * max(1, abs(b["dbeta"][j]))


@pytest.mark.parametrize("rows,cols", [(5, 17), (3, 256), (9, 1000)])
def test_backward_matches_torch_autograd(rows, cols):
    eps = 1e-5
    x = _rand((rows, cols), 61)
    res = _rand((rows, cols), 62)
    dy = _rand((rows, cols), 63)
    gamma, beta = _ln_params(cols, 64)
    r = oracle.ln_fwd(x, res, gamma, beta, eps, io="f64")
    b = oracle.ln_bwd(dy, r["res_out"], gamma, r["mean"], r["rstd"], io="f64")
    xt = torch.tensor(x, requires_grad=True)
    rt = torch.tensor(res, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    bt = torch.tensor(beta, requires_grad=True)
    y = torch.nn.functional.layer_norm(xt + rt, (cols,), gt, bt, eps)
    (y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(r["out"], y.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(b["dx"], xt.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(b["dx"], rt.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(b["dgamma"], gt.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b["dbeta"], bt.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_hw4_and_slides_forms_agree():
    g = json.load(open(os.path.join(GOLDEN, "backward_forms_agree.json")))
    rows, cols, eps = 6, 64, 1e-5
    x = _rand((rows, cols), 71)
    dy = _rand((rows, cols), 72)
    gamma, beta = _ln_params(cols, 73)
    r = oracle.ln_fwd(x, None, gamma, beta, eps, io="f64")
    hw4 = oracle.ln_bwd(dy, r["res_out"], gamma, r["mean"], r["rstd"], io="f64")["dx"]
    slides = oracle.ln_bwd_dx_slides(dy, r["res_out"], gamma, r["mean"], r["rstd"])
    scale = np.max(np.abs(hw4))
    assert np.max(np.abs(hw4 - slides)) <= g["tolerance_used_here_relative"] * scale


def test_backward_invariants():
    g = json.load(open(os.path.join(GOLDEN, "sum_dx_zero.json")))
    rows, cols, eps = 8, 129, 1e-3  # large eps so the second invariant is not trivially 0
    x = _rand((rows, cols), 81, scale=0.05)
    dy = _rand((rows, cols), 82)
    gamma, beta = _ln_params(cols, 83)
    r = oracle.ln_fwd(x, None, gamma, beta, eps, io="f64")
    b = oracle.ln_bwd(dy, r["res_out"], gamma, r["mean"], r["rstd"], io="f64")
    scale = np.max(np.abs(b["dx"]))
    np.testing.assert_allclose(b["dx"].sum(axis=1), g["per_row_sum_of_dx"], atol=1e-12 * scale * cols)
    # Derived here: sum_i dx_i xhat_i = rstd * sum(g xhat) * eps / (var + eps).
    xhat = (x - r["mean"][:, None]) * r["rstd"][:, None]
    var = x.var(axis=1)
    sgx = (gamma[None, :] * dy * xhat).sum(axis=1)
    lhs = (b["dx"] * xhat).sum(axis=1)
    rhs = r["rstd"] * sgx * eps / (var + eps)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-9, atol=1e-12 * scale * cols)
    assert np.max(np.abs(rhs)) > 1e-3


def test_backward_single_row_column_gradients():
    cols, eps = 40, 1e-5
    x = _rand((1, cols), 91)
    dy = _rand((1, cols), 92)
    gamma, beta = _ln_params(cols, 93)
    r = oracle.ln_fwd(x, None, gamma, beta, eps, io="f64")
    b = oracle.ln_bwd(dy, r["res_out"], gamma, r["mean"], r["rstd"], io="f64")
    xhat = (x[0] - r["mean"][0]) * r["rstd"][0]
    np.testing.assert_array_equal(b["dgamma"], dy[0] * xhat)
    np.testing.assert_array_equal(b["dbeta"], dy[0])


def test_column_sums_are_row_ordered_sums():
    """dgamma/dbeta at a size where the threaded column loop matters, against NumPy."""
    rows, cols = 1000, 300
    x = _rand((rows, cols), 101)
    dy = _rand((rows, cols), 102)
    gamma, beta = _ln_params(cols, 103)
    r = oracle.ln_fwd(x, None, gamma, beta, 1e-5, io="f64")
    b = oracle.ln_bwd(dy, r["res_out"], gamma, r["mean"], r["rstd"], io="f64", threads=3)
    xhat = (x - r["mean"][:, None]) * r["rstd"][:, None]
    np.testing.assert_allclose(b["dgamma"], (dy * xhat).sum(axis=0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b["dbeta"], dy.sum(axis=0), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------------------
# Rounding pins
# ----------------------------------------------------------------------------------------
def test_bf16_rounding_ties_and_library():
    one = 1.0
    cases = {
        one + 2.0 ** -8: 1.0,                         # exact tie -> even (1.0)
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,         # exact tie -> even (1 + 2^-6)
        one + 2.0 ** -8 + 2.0 ** -40: one + 2.0 ** -7,  # just above the tie -> up
        -(one + 2.0 ** -8): -1.0,
        100.25: 100.0,                                # spacing 0.5 at 100: tie -> even
        100.75: 101.0,
        3.0e38: 226 * 2.0 ** 120,                     # spacing 2^120 near 3e38
        3.4e38: np.inf,                               # above (max + half spacing)
        2.0 ** -135: 0.0,                             # below half the subnormal spacing
        3 * 2.0 ** -134: 2.0 ** -132,                 # subnormal tie -> even
    }
    got = oracle.round_io(np.array(list(cases)), "bf16")
    np.testing.assert_array_equal(got, np.array(list(cases.values())))
    np.testing.assert_array_equal(numpy_ref.round_bf16(np.array(list(cases))), got)
    # Random fp32-representable values: torch's fp32 -> bf16 cast is round-to-nearest-even.
    v = np.random.default_rng(7).normal(0, 3, 20000).astype(np.float32)
    v = np.concatenate([v, v * 1e-30, v * 1e30])
    ref = torch.tensor(v).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_io(v.astype(np.float64), "bf16"), ref)


def test_f32_rounding_matches_numpy_cast():
    v = np.random.default_rng(8).normal(0, 1, 5000) * 10.0 ** np.random.default_rng(9).integers(-30, 30, 5000)
    np.testing.assert_array_equal(oracle.round_io(v, "f32"), v.astype(np.float32).astype(np.float64))


# ----------------------------------------------------------------------------------------
# The C oracle and its NumPy twin agree
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(1, 1), (4, 3), (33, 130), (17, 1000)])
def test_c_oracle_matches_numpy_twin(io, rows, cols):
    x = oracle.round_io(_rand((rows, cols), 111, loc=2.0), io)
    res = oracle.round_io(_rand((rows, cols), 112), io)
    dy = oracle.round_io(_rand((rows, cols), 113), io)
    gamma, beta = (oracle.round_io(p, io) for p in _ln_params(cols, 114))
    c = oracle.ln_fwd(x, res, gamma, beta, 1e-5, io=io)
    n = numpy_ref.ln_fwd(x, res, gamma, beta, 1e-5, io=io)
    np.testing.assert_array_equal(c["res_out"], n["res_out"])
    np.testing.assert_allclose(c["mean"], n["mean"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(c["rstd"], n["rstd"], rtol=1e-12)
    atol = 1e-12 if io == "f64" else 0
    rtol = 0 if io == "f64" else 2.0 ** -7  # a value within 1e-15 of a tie may round apart
    np.testing.assert_allclose(c["out"], n["out"], rtol=rtol, atol=atol)
    cb = oracle.ln_bwd(dy, c["res_out"], gamma, c["mean"], c["rstd"], io=io)
    nb = numpy_ref.ln_bwd(dy, c["res_out"], gamma, c["mean"], c["rstd"], io=io)
    for k in ("dx", "dgamma", "dbeta"):
        np.testing.assert_allclose(cb[k], nb[k], rtol=max(rtol, 1e-11), atol=1e-11)


# ----------------------------------------------------------------------------------------
# The pins catch planted mistakes (mistakes planted in a copy of the NumPy twin, on the CPU)
# ----------------------------------------------------------------------------------------
def _mutant_bwd(kind):
    def bwd(dy, xr, gamma, mean, rstd):
        m = dy.shape[1]
        xhat = (xr - mean[:, None]) * rstd[:, None]
        g = gamma[None, :] * dy
        sg = g.sum(axis=1, keepdims=True)
        sgx = (g * xhat).sum(axis=1, keepdims=True)
        if kind == "dropped_term":
            dx = rstd[:, None] * (g - sg / m)
        elif kind == "wrong_sign":
            dx = rstd[:, None] * (g - (sg - xhat * sgx) / m)
        elif kind == "transposed_gamma":
            dx = rstd[:, None] * (gamma[::-1][None, :] * dy - (sg + xhat * sgx) / m)
        else:
            raise ValueError(kind)
        return dx
    return bwd


@pytest.mark.parametrize("kind", ["dropped_term", "wrong_sign", "transposed_gamma"])
def test_pins_catch_planted_mistakes(kind):
    rows, cols, eps = 3, 5, 1e-5
    x = _rand((rows, cols), 121)
    dy = _rand((rows, cols), 122)
    gamma, beta = _ln_params(cols, 123)
    r = numpy_ref.ln_fwd(x, None, gamma, beta, eps)
    bad = _mutant_bwd(kind)(dy, r["res_out"], gamma, r["mean"], r["rstd"])
    xt = torch.tensor(x, requires_grad=True)
    y = torch.nn.functional.layer_norm(xt, (cols,), torch.tensor(gamma), torch.tensor(beta), eps)
    (y * torch.tensor(dy)).sum().backward()
    assert np.max(np.abs(bad - xt.grad.numpy())) > 1e-3


def test_pins_catch_unbiased_variance_and_eps_placement():
    row = np.array([[1000.0, 1001.0]])
    g = json.load(open(os.path.join(GOLDEN, "two_values_1000_1001.json")))
    unbiased = row.var(axis=1, ddof=1)[0]
    assert unbiased != g["var"]
    # eps outside the square root would change rstd measurably at this variance.
    eps = 1e-2
    r = oracle.ln_fwd(row, None, np.ones(2), np.zeros(2), eps, io="f64")
    assert abs(r["rstd"][0] - 1.0 / (np.sqrt(g["var"]) + eps)) > 1e-4
    assert r["rstd"][0] == 1.0 / np.sqrt(g["var"] + eps)
