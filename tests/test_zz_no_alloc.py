"""The allocation-free backward, ln_bwd_bf16_noalloc, against the regular ln_bwd_bf16.

Callers that cannot allocate device memory while they run (a serving process that reserved
its memory budget at start-up, a plugin whose host framework owns all device allocations)
use ln_bwd_bf16_noalloc, which keeps its scratch in a fixed array inside the library.  This
test calls it through the C ABI twice in a row -- the second call finds the array holding
the first call's leftovers -- and checks each result against the regular entry point within
the bf16 tolerance the parity tests use.  This file is named so that pytest collects it
last; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import layernorm_ln_fwd_gb300 as ln
import lnparity as P
from layernorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("rows,cols", [(8192, 768), (300, 1001)])
def test_noalloc_backward_matches_regular_backward_twice(rows, cols):
    L = ln.lib()
    stream = torch.cuda.current_stream()
    for seed in (11, 12):  # two calls in a row, different data
        inp = synth.make_inputs(rows, cols, "bf16", seed=seed)
        d = P.to_device(inp)
        out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], synth.EPS)
        dx_ref, dg_ref, db_ref = ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd)
        dx = torch.full_like(dx_ref, float("nan"))
        dg = torch.full_like(dg_ref, float("nan"))
        db = torch.full_like(db_ref, float("nan"))
        st = L.ln_bwd_bf16_noalloc(_p(d["dy"]), _p(res_out), _p(d["gamma"]), _p(mean),
                                   _p(rstd), _p(dx), _p(dg), _p(db), rows, cols,
                                   ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, ln.STATUS.get(st, st)
        torch.cuda.synchronize()
        for name, got, ref in (("dx", dx, dx_ref), ("dgamma", dg, dg_ref),
                               ("dbeta", db, db_ref)):
            P.compare(name, P.to64(got), P.to64(ref), "bf16")


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = ln.lib()
    p = ctypes.c_void_p(256)  # never touched: the size check comes first
    # 65536 x 16384 needs far more than LN_NOALLOC_SCRATCH_BYTES of partial sums.
    assert L.ln_bwd_bf16_noalloc(p, p, p, p, p, p, p, p, 65536, 16384, None) == 3
