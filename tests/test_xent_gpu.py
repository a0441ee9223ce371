"""Parity of the fused cross-entropy kernel (called through the C ABI) with the float64
oracle ("Accelerating Transformer on GPU (I)", section 5.2): losses (fp32, 2e-5 relative
above 1 as for the other fp32 statistics) and the gradient dloss * (q - p) (fp32 2e-5,
bf16 2 ulps), with and without label smoothing, in place over the logits, for vocabulary
widths that are and are not 16-byte multiples (GPT-2's 50257, llm.c's padded 50304), on
both forms of the kernel (rows staged in shared memory, rows streamed through L2), and at
the GPT-2-small classifier size (8 x 1024 rows) on every element."""
import numpy as np
import pytest
import torch

import layernorm_ln_fwd_gb300 as ln
import lnparity as P
import oracle
from layernorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu


def case(rows, V, dtype, seed, spread=2.0):
    inp = synth.make_inputs(rows, V, dtype, seed=seed, x=("normal", 0.0, spread))
    g = torch.Generator().manual_seed(seed)
    t = torch.randint(0, V, (rows,), generator=g, dtype=torch.int32)
    return inp["x"], t


def check(x, t, alpha, dloss, dtype, in_place=False):
    d_x = x.cuda()
    losses, dlogits = ln.xent(d_x, t.cuda(), alpha, dloss, in_place=in_place)
    torch.cuda.synchronize()
    ref = oracle.xent(P.to64(x), t.numpy(), alpha, dloss, io=dtype)
    infos = [P.compare("loss", P.to64(losses), ref["loss"], "f32"),
             P.compare("dx", P.to64(dlogits), ref["dx"], dtype)]
    if in_place:
        assert dlogits.data_ptr() == d_x.data_ptr()
    return infos


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 8, 256, 1000, 1001, 4096, 50257, 50304])
@pytest.mark.parametrize("alpha", [0.0, 0.1])
def test_widths_against_oracle(dtype, V, alpha):
    rows = 64 if V < 10000 else 24
    x, t = case(rows, V, dtype, seed=V)
    check(x, t, alpha, 1.0 / rows, dtype)


@pytest.mark.parametrize("dtype,V", [("bf16", 56320), ("bf16", 65536), ("f32", 24576),
                                     ("f32", 50304)])
def test_staged_and_streaming_forms(dtype, V):
    """Rows of 16-byte vectors that fit twice in shared memory are staged whole (bf16 56320:
    2 x 110 KB; fp32 24576: 2 x 96 KB); wider ones stream through L2 (bf16 65536, fp32
    50304).  Both forms against the oracle, in place and not."""
    x, t = case(12, V, dtype, seed=V + 1)
    check(x, t, 0.1, 1.0 / 12, dtype)
    check(x, t, 0.0, 1.0, dtype, in_place=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_in_place_gradient(dtype):
    x, t = case(40, 50304, dtype, seed=3)
    check(x, t, 0.1, 1.0, dtype, in_place=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_losses_only_and_gradient_only(dtype):
    x, t = case(16, 2048, dtype, seed=4)
    d_x, d_t = x.cuda(), t.cuda()
    losses, g = ln.xent(d_x, d_t, 0.1, 1.0, want_grad=False)
    assert g is None
    ref = oracle.xent(P.to64(x), t.numpy(), 0.1, 1.0, io=dtype)
    torch.cuda.synchronize()
    P.compare("loss", P.to64(losses), ref["loss"], "f32")
    losses, g = ln.xent(d_x, d_t, 0.1, 1.0, want_losses=False)
    torch.cuda.synchronize()
    assert losses is None
    P.compare("dx", P.to64(g), ref["dx"], dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_large_logits_do_not_overflow(dtype):
    x, t = case(8, 1024, dtype, seed=5, spread=200.0)
    check(x, t, 0.2, 1.0, dtype)


def test_gpt2_classifier_size_every_element():
    """8 x 1024 tokens over llm.c's padded GPT-2 vocabulary of 50304, bf16 logits, mean loss
    (dloss = 1 / rows), label smoothing 0.1; repeatable bit for bit."""
    rows, V = 8192, 50304
    x, t = case(rows, V, "bf16", seed=0)
    infos = check(x, t, 0.1, 1.0 / rows, "bf16")
    assert all(i["n_over_stated"] == 0 for i in infos)
    d_x, d_t = x.cuda(), t.cuda()
    a = ln.xent(d_x, d_t, 0.1, 1.0 / rows)
    b = ln.xent(d_x, d_t, 0.1, 1.0 / rows)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_invalid_arguments():
    x = torch.zeros(4, 8, device="cuda")
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(ln.LnError):
        ln.xent(x, t, alpha=1.5)
    with pytest.raises(ln.LnError):
        ln.xent(x, t, want_losses=False, want_grad=False)
