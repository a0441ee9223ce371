"""Pins for the float64 oracle of the fused cross-entropy with label smoothing (CPU only).

"Accelerating Transformer on GPU (I)", section 5.2: p = (1 - alpha) onehot(t) + alpha / V
(the page notes this is PyTorch's label_smoothing convention, not the eps / (V - 1) one),
q = softmax(x), loss = -sum p log q = log Z + m - [(1 - alpha) x_t + (alpha / V) sum x], and
the gradient is q - p (times the upstream dloss).  Pinned to torch's float64
cross_entropy(label_smoothing=alpha) and its autograd, the NumPy twin (written as the
page's -sum p log q), closed forms (uniform logits give log V; alpha = 0 gives
log Z + m - x_t; the gradient sums to zero), finite differences, and planted mistakes (the
eps / (V - 1) convention, the sign, the missing max).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import numpy_ref


def _case(rows, V, seed, spread=3.0):
    rng = np.random.default_rng(seed)
    return rng.normal(0, spread, (rows, V)), rng.integers(0, V, rows)


@pytest.mark.parametrize("alpha", [0.0, 0.1, 0.5])
def test_matches_torch_cross_entropy(alpha):
    x, t = _case(7, 53, 1)
    r = oracle.xent(x, t, alpha)
    xt = torch.tensor(x, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(xt, torch.tensor(t), reduction="none",
                                             label_smoothing=alpha)
    np.testing.assert_allclose(r["loss"], loss.detach().numpy(), rtol=1e-13, atol=1e-13)
    loss.sum().backward()
    np.testing.assert_allclose(r["dx"], xt.grad.numpy(), rtol=1e-12, atol=1e-15)
    # dloss scales the gradient (a mean over rows: dloss = 1 / rows).
    r2 = oracle.xent(x, t, alpha, dloss=1.0 / 7)
    np.testing.assert_allclose(r2["dx"], xt.grad.numpy() / 7, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("io", ["f64", "f32", "bf16"])
def test_c_oracle_matches_numpy_twin(io):
    x, t = _case(6, 300, 2)
    x = oracle.round_io(x, io)
    a = oracle.xent(x, t, 0.1, 0.25, io=io)
    b = numpy_ref.xent(x, t, 0.1, 0.25, io=io)
    np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-12)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(b["dx"]), 1e-300))) -
                  {"f64": 40, "f32": 23, "bf16": 7}[io])
    assert np.all(np.abs(a["dx"] - b["dx"]) <= ulp)


def test_closed_forms_and_invariants():
    V = 64
    r = oracle.xent(np.full((3, V), 2.5), np.array([0, 5, 63]), 0.3)
    np.testing.assert_allclose(r["loss"], np.log(V), rtol=1e-14)
    x, t = _case(5, V, 3)
    r0 = oracle.xent(x, t, 0.0)
    m = x.max(axis=1)
    lz = np.log(np.exp(x - m[:, None]).sum(axis=1))
    np.testing.assert_allclose(r0["loss"], lz + m - x[np.arange(5), t], rtol=1e-13)
    r1 = oracle.xent(x, t, 0.2)
    np.testing.assert_allclose(r1["dx"].sum(axis=1), 0.0, atol=1e-15)
    # Large logits: the max is subtracted first.
    rb = oracle.xent(np.array([[1000.0, 0.0, -1000.0]]), np.array([0]), 0.0)
    assert np.isfinite(rb["loss"][0]) and abs(rb["loss"][0]) < 1e-12


def test_finite_differences():
    x, t = _case(2, 6, 4)
    alpha, h = 0.2, 1e-6
    r = oracle.xent(x, t, alpha)
    for i in range(2):
        for j in range(6):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            num = (oracle.xent(xp, t, alpha)["loss"].sum() -
                   oracle.xent(xm, t, alpha)["loss"].sum()) / (2 * h)
            assert abs(num - r["dx"][i, j]) < 1e-8


@pytest.mark.parametrize("kind", ["eps_over_v_minus_1", "sign", "no_max"])
def test_pins_catch_planted_mistakes(kind):
    x, t = _case(4, 30, 5)
    x[0, 0] = 800.0  # a large logit: only a max-shifted evaluation stays finite
    alpha = 0.1
    rows, V = x.shape
    if kind == "eps_over_v_minus_1":
        p = np.full((rows, V), alpha / (V - 1))
        p[np.arange(rows), t] = 1.0 - alpha
    else:
        p = np.full((rows, V), alpha / V)
        p[np.arange(rows), t] += 1.0 - alpha
    with np.errstate(all="ignore"):
        if kind == "no_max":
            q = np.exp(x) / np.exp(x).sum(axis=1, keepdims=True)
        else:
            z = x - x.max(axis=1, keepdims=True)
            q = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
        bad = p - q if kind == "sign" else q - p
    xt = torch.tensor(x, requires_grad=True)
    torch.nn.functional.cross_entropy(xt, torch.tensor(t), reduction="sum",
                                      label_smoothing=alpha).backward()
    assert not np.allclose(bad, xt.grad.numpy(), atol=1e-6)
    np.testing.assert_allclose(oracle.xent(x, t, alpha)["dx"], xt.grad.numpy(), rtol=1e-12,
                               atol=1e-15)
