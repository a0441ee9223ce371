"""The allocation-free backward, ln_bwd_bf16_noalloc, against the regular ln_bwd_bf16.

Callers that cannot allocate device memory while they run (a serving process that reserved
its memory budget at start-up, a plugin whose host framework owns all device allocations)
use ln_bwd_bf16_noalloc, which keeps its scratch in a fixed array inside the library.  It
runs the same plan and kernels as ln_bwd_bf16, in the same summation order, so its results
must be bit for bit those of ln_bwd_bf16; they are also checked against the float64 oracle.
Each shape is called twice in a row through the C ABI: the second call relies on the first
having left the shared array all zero.  After a bounded wait that ran out, ln_device_check
must zero the array again so that the next call is correct.  This file is named so that
pytest collects it last; it also passes on its own in a fresh process.
"""
import ctypes
import os

import pytest
import torch

import layernorm_ln_fwd_gb300 as ln
import lnparity as P
from layernorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(d, res_out, mean, rstd, stream):
    rows, cols = d["dy"].shape
    dx = torch.full_like(d["dy"], float("nan"))
    dg = torch.full_like(d["gamma"], float("nan"))
    db = torch.full_like(d["gamma"], float("nan"))
    st = ln.lib().ln_bwd_bf16_noalloc(_p(d["dy"]), _p(res_out), _p(d["gamma"]), _p(mean),
                                      _p(rstd), _p(dx), _p(dg), _p(db), rows, cols,
                                      ctypes.c_void_p(stream.cuda_stream))
    return st, dx, dg, db


@pytest.mark.parametrize("rows,cols", [(8192, 768), (8192, 1280), (300, 1001), (37, 4104)])
def test_noalloc_backward_matches_regular_backward_twice(rows, cols):
    """(8192, 768), (8192, 1280): the warp-per-row kernel; (300, 1001): rows that are not
    16-byte multiples, the scalar kernel; (37, 4104): the block-per-row kernel."""
    stream = torch.cuda.current_stream()
    for seed in (11, 12):  # two calls in a row, different data
        inp = synth.make_inputs(rows, cols, "bf16", seed=seed)
        d = P.to_device(inp)
        out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], synth.EPS)
        dx_ref, dg_ref, db_ref = ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd)
        st, dx, dg, db = _noalloc(d, res_out, mean, rstd, stream)
        assert st == 0, ln.STATUS.get(st, st)
        # The block-per-row kernel (aligned rows wider than 1280 bf16 columns) hands its
        # column sums' finish to a second, dependent launch.
        assert ln.last_launch_count() == (2 if cols > 1280 and cols % 8 == 0 else 1)
        torch.cuda.synchronize()
        for name, got, ref in (("dx", dx, dx_ref), ("dgamma", dg, dg_ref),
                               ("dbeta", db, db_ref)):
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), name
        ref = P.run_oracle(inp, synth.EPS)
        for name, got in (("dx", dx), ("dgamma", dg), ("dbeta", db)):
            P.compare(name, P.to64(got), ref[name], "bf16",
                      extra=ref["_colsum"].get(name))


def test_noalloc_recovers_after_a_timeout():
    """The finishers' bounded wait is made to run out (a 2 ms limit on a word nothing
    writes): the call returns, ln_device_check reports LN_ETIMEOUT and zeroes the fixed
    array, and the next call matches ln_bwd_bf16 bit for bit."""
    rows, cols = 512, 768
    inp = synth.make_inputs(rows, cols, "bf16", seed=13)
    d = P.to_device(inp)
    stream = torch.cuda.current_stream()
    out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], synth.EPS)
    check_mode = os.environ.get("LN_CHECK", "0") not in ("", "0")
    L = ln.lib()
    L.ln_debug_wait_test(2000)
    try:
        st, _, _, _ = _noalloc(d, res_out, mean, rstd, stream)
        if check_mode:  # the call synchronises and reports the timeout itself
            assert st == 5
        else:
            assert st == 0
            assert ln.device_check() == 5
    finally:
        L.ln_debug_wait_test(0)
    assert ln.device_check() == 0
    dx_ref, dg_ref, db_ref = ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd)
    st, dx, dg, db = _noalloc(d, res_out, mean, rstd, stream)
    assert st == 0
    torch.cuda.synchronize()
    for got, ref in ((dx, dx_ref), (dg, dg_ref), (db, db_ref)):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = ln.lib()
    p = ctypes.c_void_p(256)  # never touched: the size check comes first
    # 65536 x 16384 needs far more than LN_NOALLOC_SCRATCH_BYTES of partial sums.
    assert L.ln_bwd_bf16_noalloc(p, p, p, p, p, p, p, p, 65536, 16384, None) == 3
    assert L.ln_last_launch_count() == 0
    # The advertised rule: a problem whose workspace bound fits the array is accepted (the
    # 8192 x 768 call above is one).
    assert ln.workspace_bytes(8192, 768) <= 16 << 20
