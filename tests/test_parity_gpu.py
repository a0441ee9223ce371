"""Parity of the CUDA path (called through the C ABI) with the float64 oracle.

Small shapes run the oracle on every element; the five full-size workloads (and the
benchmark's three other widths) compare every row (a sample of the 262144-row one) element
by element and dgamma/dbeta over all rows, in the launch configuration the benchmark uses;
rows wider than one warp's registers (2 or 4 warps per row) are swept over thirteen widths.
Tolerances are stated in ``lnparity``.
"""
import os

import numpy as np
import pytest
import torch

import layernorm_ln_fwd_gb300 as ln
import lnparity as P
import oracle
from layernorm_ln_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = synth.EPS

COLS = [1, 2, 3, 8, 31, 32, 33, 127, 128, 129, 767, 768, 1000, 1001, 1023, 1024, 1025, 1280,
        2048, 2056, 4096, 8191, 8192, 16384]
ROWS = [1, 7, 300]
# dgamma/dbeta columns allowed over the bare stated bound (each within the column-sum
# allowance): columns whose terms cancel to almost zero, where the bare bound is a few bf16
# ulps of a tiny value.
MAX_COLUMNS_OVER_STATED = 5


@pytest.fixture(autouse=True)
def _auto_path():
    ln.force_path(ln.PATH_AUTO)
    yield
    ln.force_path(ln.PATH_AUTO)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("rows", ROWS)
def test_shapes_against_oracle(dtype, rows, cols):
    inp = synth.make_inputs(rows, cols, dtype, seed=rows * 100003 + cols)
    gpu = P.run_gpu(inp, EPS)
    ref = P.run_oracle(inp, EPS)
    P.compare_all(gpu, ref, dtype, conditioned=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
def test_backward_on_identical_stored_inputs(dtype, cols):
    """The backward alone, fed the same stored inputs on both sides (the oracle forward's
    res_out, and its mean and rstd rounded to fp32): no conditioning term is needed."""
    rows = 300
    inp = synth.make_inputs(rows, cols, dtype, seed=cols + 17)
    st = P.stored_stats_inputs(inp, EPS)
    td = synth.torch_dtype(dtype)
    dev = lambda a, t=td: torch.tensor(a).to(t).cuda()  # noqa: E731  (exact casts)
    dx, dg, db = ln.bwd(inp["dy"].cuda(), dev(st["res_out"]), inp["gamma"].cuda(),
                        dev(st["mean"], torch.float32), dev(st["rstd"], torch.float32))
    torch.cuda.synchronize()
    dy64 = P.to64(inp["dy"])
    b = oracle.ln_bwd(dy64, st["res_out"], P.to64(inp["gamma"]), st["mean"], st["rstd"],
                      io=dtype)
    allow = P.colsum_allowance(dy64, (st["res_out"] - st["mean"][:, None]) * st["rstd"][:, None])
    P.compare("dx", P.to64(dx), b["dx"], dtype)
    P.compare("dgamma", P.to64(dg), b["dgamma"], dtype, extra=allow["dgamma"])
    P.compare("dbeta", P.to64(db), b["dbeta"], dtype, extra=allow["dbeta"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", [ln.PATH_WARP, ln.PATH_BLOCK, ln.PATH_SCALAR])
@pytest.mark.parametrize("rows,cols", [(5, 64), (37, 768), (64, 1024), (19, 1000), (9, 4104)])
def test_every_kernel_family(dtype, path, rows, cols):
    if dtype == "bf16" and cols == 1000:
        cols = 1000 - 8  # keep bf16 rows 16-byte multiples so the vector paths apply
    ln.force_path(path)
    inp = synth.make_inputs(rows, cols, dtype, seed=7 + path)
    P.compare_all(P.run_gpu(inp, EPS), P.run_oracle(inp, EPS), dtype, conditioned=True)


# Rows wider than one warp's share of registers go to the backward tile kernel with 2 or 4
# warps per row (bf16 1288-4096 columns, fp32 1028-2048) and, at bf16 2056-3072 columns, to
# the forward tile kernel with 4 warps per row; 2503 rows give every block several tiles and
# a ragged last tile at every rows-per-tile the plans pick (7, 5, 3, 2).
WIDE_TILE = [("bf16", 1288), ("bf16", 1536), ("bf16", 1600), ("bf16", 2048), ("bf16", 2056),
             ("bf16", 2560), ("bf16", 3072), ("bf16", 4096), ("f32", 1028), ("f32", 1280),
             ("f32", 1284), ("f32", 1600), ("f32", 2048)]


@pytest.mark.parametrize("dtype,cols", WIDE_TILE)
def test_rows_shared_by_several_warps(dtype, cols):
    """Every element against the oracle: the bare stated tolerances, except that a few
    dgamma/dbeta columns whose terms cancel to almost zero may use the column-sum allowance;
    and the backward bitwise repeatable (the warps of a row add their row sums in warp
    order)."""
    inp = synth.make_inputs(2503, cols, dtype, seed=cols + 3)
    gpu = P.run_gpu(inp, EPS)
    infos = P.compare_all(gpu, P.run_oracle(inp, EPS), dtype)
    over = {i["name"]: i["n_over_stated"] for i in infos if i["n_over_stated"]}
    assert set(over) <= {"dgamma", "dbeta"}, over
    assert all(n <= MAX_COLUMNS_OVER_STATED for n in over.values()), over
    d = P.to_device(inp)
    for _ in range(2):
        dx2, dg2, db2 = ln.bwd(d["dy"], gpu["res_out"], d["gamma"], gpu["mean"], gpu["rstd"])
        torch.cuda.synchronize()
        assert torch.equal(dx2, gpu["dx"]) and torch.equal(dg2, gpu["dgamma"])
        assert torch.equal(db2, gpu["dbeta"])


@pytest.mark.parametrize("cols", [1536, 2560, 3072])
def test_rows_shared_by_several_warps_long_chains(cols):
    """bf16 with more than 65536 rows: the per-lane column sums are compensated (2 warps per
    row with 3 and 5 vectors per lane; at 3072 columns the block-per-row kernel); rows
    compared on a sample, dgamma/dbeta over all rows."""
    rows = 65600
    inp = synth.make_inputs(rows, cols, "bf16", seed=cols)
    gpu = P.run_gpu(inp, EPS)
    rng = np.random.default_rng(2)
    rows_idx = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 254, replace=False)]))
    infos = P.compare_all(gpu, P.run_oracle(inp, EPS, rows_idx=rows_idx), "bf16",
                          rows_idx=rows_idx)
    ref_p = P.oracle_dparams(inp, EPS)
    for k in ("dgamma", "dbeta"):
        infos.append(P.compare(k, P.to64(gpu[k]), ref_p[k], "bf16", extra=ref_p["_colsum"][k]))
    over = {i["name"]: i["n_over_stated"] for i in infos if i["n_over_stated"]}
    assert set(over) <= {"dgamma", "dbeta"}, over
    assert all(n <= MAX_COLUMNS_OVER_STATED for n in over.values()), over


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [768, 1000, 2560, 8192])
def test_plain_layernorm_without_residual(dtype, cols):
    inp = synth.make_inputs(33, cols, dtype, seed=3)
    gpu = P.run_gpu(inp, EPS, has_res=False)
    ref = P.run_oracle(inp, EPS, has_res=False)
    P.compare_all(gpu, ref, dtype)
    # res_out receives a copy of x.
    assert torch.equal(gpu["res_out"].cpu(), inp["x"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward_without_res_out(dtype):
    inp = synth.make_inputs(40, 1280, dtype, seed=4)
    gpu = P.run_gpu(inp, EPS, write_res=False)
    assert "res_out" not in gpu
    ref = P.run_oracle(inp, EPS)
    for k in ("out", "mean", "rstd"):
        P.compare(k, P.to64(gpu[k]), ref[k], dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [768, 8192])
def test_unaligned_pointers_take_the_scalar_kernel(dtype, cols):
    rows = 23
    inp = synth.make_inputs(rows, cols, dtype, seed=5)
    td = synth.torch_dtype(dtype)

    def shifted(t):  # same values, data pointer off by one element (not 16-byte aligned)
        buf = torch.empty(t.numel() + 1, dtype=td, device="cuda")
        v = buf[1:].view(t.shape)
        v.copy_(t.cuda())
        return v

    d = {k: shifted(v) for k, v in inp.items()}
    assert d["x"].data_ptr() % 16 != 0
    out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], EPS,
                                      out=shifted(inp["x"]), res_out=shifted(inp["x"]))
    dx, dg, db = ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd, dx=shifted(inp["x"]))
    torch.cuda.synchronize()
    gpu = {"out": out, "res_out": res_out, "mean": mean, "rstd": rstd, "dx": dx,
           "dgamma": dg, "dbeta": db}
    P.compare_all(gpu, P.run_oracle(inp, EPS), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_caller_owned_workspace(dtype):
    rows, cols = 300, 1280
    inp = synth.make_inputs(rows, cols, dtype, seed=6)
    ws = torch.zeros(ln.workspace_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    assert ws.data_ptr() % 256 == 0
    ref = P.run_oracle(inp, EPS)
    for _ in range(2):  # each call leaves the workspace zeroed, so it can be reused
        P.compare_all(P.run_gpu(inp, EPS, workspace=ws), ref, dtype)
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ln.LnError) as e:
        P.run_gpu(inp, EPS, workspace=small)
    assert e.value.status == 6


def test_workspace_is_left_zero_and_serves_every_shape():
    """One caller-owned workspace, backwards of several shapes and kernel families in turn:
    each result matches the oracle and each call leaves every workspace byte at zero (the
    finish reads the partial sums as they land, taking a zero word for one not yet written,
    so a stale partial left behind would be taken for the next call's)."""
    cases = [("f32", 300, 1024, ln.PATH_AUTO), ("bf16", 37, 768, ln.PATH_AUTO),
             ("bf16", 9, 4104, ln.PATH_BLOCK), ("f32", 5, 8191, ln.PATH_AUTO),
             ("bf16", 7, 1001, ln.PATH_SCALAR), ("f32", 300, 1024, ln.PATH_AUTO)]
    nbytes = max(ln.workspace_bytes(r, c) for _, r, c, _ in cases)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for i, (dtype, rows, cols, path) in enumerate(cases):
        ln.force_path(path)
        inp = synth.make_inputs(rows, cols, dtype, seed=40 + i)
        P.compare_all(P.run_gpu(inp, EPS, workspace=ws), P.run_oracle(inp, EPS), dtype,
                      conditioned=True)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws)) == 0, (dtype, rows, cols, path)


@pytest.mark.parametrize("dtype,rows,cols,path", [
    ("f32", 300, 1024, ln.PATH_AUTO),    # warp per row, compensated (hi, lo) partials
    ("bf16", 300, 768, ln.PATH_AUTO),    # warp per row, plain partials
    ("bf16", 9, 4104, ln.PATH_BLOCK),
    ("f32", 64, 4104, ln.PATH_BLOCK),
    ("f32", 37, 1001, ln.PATH_AUTO),     # scalar (unaligned rows)
])
def test_nan_in_dy_propagates_and_the_finish_completes(dtype, rows, cols, path):
    """A NaN in dy makes its row of dx and its column of dgamma and dbeta NaN, as in the
    oracle, and everything else still matches.  The NaN also reaches the stored partial sums
    -- as the negated compensation of a Kahan sum its bits can be 0xffffffff, the one pattern
    the partial encoding must move off the zero word -- and the finish must still see every
    partial as written (no timeout)."""
    ln.force_path(path)
    inp = synth.make_inputs(rows, cols, dtype, seed=77)
    dy = inp["dy"].clone()
    dy[rows // 2, 3] = float("nan")
    inp["dy"] = dy
    gpu = P.run_gpu(inp, EPS)
    assert ln.device_check() == 0
    ref = P.run_oracle(inp, EPS)
    io = dtype
    for name in ("dx", "dgamma", "dbeta"):
        g, r = P.to64(gpu[name]), ref[name]
        assert np.array_equal(np.isnan(g), np.isnan(r)), name
        assert np.isnan(r).any(), name
        ok = ~np.isnan(r)
        extra = None
        for part in (ref["_conditioning"].get(name), ref["_colsum"].get(name)):
            if part is not None:
                extra = part if extra is None else extra + part
        P.compare(name, g[ok], r[ok], io, extra=None if extra is None else extra[ok])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_rows(dtype):
    td = synth.torch_dtype(dtype)
    x = torch.empty(0, 64, dtype=td, device="cuda")
    g = torch.ones(64, dtype=td, device="cuda")
    out, res_out, mean, rstd = ln.fwd(x, x, g, g, EPS)
    assert out.shape == (0, 64)
    dgamma = torch.full((64,), 7.0, dtype=td, device="cuda")
    dbeta = torch.full((64,), 7.0, dtype=td, device="cuda")
    ln.bwd(x, x, g, mean, rstd, dgamma=dgamma, dbeta=dbeta)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dgamma) == 0 and torch.count_nonzero(dbeta) == 0


def test_too_wide_rows_are_rejected():
    x = torch.zeros(2, ln.MAX_COLS + 8, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(ln.MAX_COLS + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ln.LnError) as e:
        ln.fwd(x, None, g, g)
    assert e.value.status == 3


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(8192, 768), (4096, 8192), (2000, 1001)])
def test_integer_dy_gives_exact_dbeta(dtype, rows, cols):
    """With dy integer-valued the column sums of dy are exact in fp32, so dbeta must match
    the oracle bit for bit whatever the order of the additions."""
    inp = synth.make_inputs(rows, cols, dtype, seed=8, dy=("int", -2, 2))
    gpu = P.run_gpu(inp, EPS)
    ref = P.oracle_dparams(inp, EPS)
    np.testing.assert_array_equal(P.to64(gpu["dbeta"]), ref["dbeta"])


# The full-size workloads compared on every row (the oracle finishes them in seconds); the
# 262144-row fp32 workload on a sample of rows (dgamma and dbeta always over all rows).
SAMPLED_WORKLOADS = {"f32_262144x1000"}


@pytest.mark.parametrize("name", list(synth.WORKLOADS) + list(synth.EXTRA_WORKLOADS))
def test_workload_full_size(name):
    """The five workloads (and the benchmark's three other widths) at full size, in the
    benchmark's launch configuration: every output element by element (all rows; a 256-row
    sample of the largest), dgamma/dbeta over all rows, and bitwise-repeatable results.
    Every output of the five workloads meets the bare stated tolerance (no element needs the
    column-sum allowance), except dgamma/dbeta of the 262144-row fp32 workload, whose sums
    over 262144 rows the allowance covers for at most MAX_COLUMNS_OVER_STATED columns; the
    other widths are held to the rule of the multi-warp tests (a few dgamma/dbeta columns
    that cancel to almost zero may use the allowance)."""
    w = synth.workload(name)
    inp = synth.workload_inputs(name, seed=0)
    gpu = P.run_gpu(inp, w.eps)
    rows_idx = None
    if name in SAMPLED_WORKLOADS:
        rng = np.random.default_rng(1)
        sample = rng.choice(w.rows, min(254, w.rows), replace=False)
        rows_idx = np.unique(np.concatenate([[0, w.rows - 1], sample]))
        ref = P.run_oracle(inp, w.eps, rows_idx=rows_idx)
        ref_p = P.oracle_dparams(inp, w.eps)
    else:
        ref = P.run_oracle(inp, w.eps)
        ref_p = {"dgamma": ref.pop("dgamma"), "dbeta": ref.pop("dbeta"),
                 "_colsum": ref["_colsum"]}
    infos = P.compare_all(gpu, ref, w.dtype, rows_idx=rows_idx)
    for k in ("dgamma", "dbeta"):
        infos.append(P.compare(k, P.to64(gpu[k]), ref_p[k], w.dtype, extra=ref_p["_colsum"][k]))
    over = {i["name"]: i["n_over_stated"] for i in infos if i["n_over_stated"]}
    allowed = ({"dgamma", "dbeta"} if name in SAMPLED_WORKLOADS or name in synth.EXTRA_WORKLOADS
               else set())
    assert set(over) <= allowed, over
    # Where the allowance is used at all, only a few columns lean on it (2 of the 1000 dgamma
    # columns at 262144 rows when this was written): more means the sums got worse.
    assert all(n <= MAX_COLUMNS_OVER_STATED for n in over.values()), over
    # Run to run: the backward gives the same bits (dgamma, dbeta and dx).
    d = P.to_device(inp)
    stable = True
    for _ in range(2):
        dx2, dg2, db2 = ln.bwd(d["dy"], gpu["res_out"], d["gamma"], gpu["mean"], gpu["rstd"])
        torch.cuda.synchronize()
        stable &= bool(torch.equal(dg2, gpu["dgamma"]) and torch.equal(db2, gpu["dbeta"])
                       and torch.equal(dx2, gpu["dx"]))
    P.report({"workload": name, "rows_compared": w.rows if rows_idx is None else len(rows_idx),
              "max_abs": {i["name"]: i["max_abs"] for i in infos},
              "worst_ratio": {i["name"]: i["worst_ratio"] for i in infos},
              "n_over_stated": {i["name"]: i["n_over_stated"] for i in infos},
              "bitwise_stable": stable})
    assert stable


def test_normalised_rows_property_at_full_size():
    """gamma = 1, beta = 0: every output row has mean ~0 and variance var/(var+eps); checked
    on all 4096 rows of the wide mean-100 workload (a property that holds at any size)."""
    w = synth.WORKLOADS["bf16_4096x8192_mean100"]
    inp = synth.workload_inputs(w.name, seed=0)
    d = P.to_device(inp)
    one = torch.ones(w.cols, dtype=torch.bfloat16, device="cuda")
    zero = torch.zeros(w.cols, dtype=torch.bfloat16, device="cuda")
    out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], one, zero, w.eps)
    o = out.double()
    s = res_out.double()
    var = s.var(dim=1, unbiased=False)
    assert float(o.mean(dim=1).abs().max()) < 2e-3  # bf16 rounding of ~1-sized outputs
    rel = (o.var(dim=1, unbiased=False) / (var / (var + w.eps)) - 1).abs().max()
    assert float(rel) < 5e-3
    np.testing.assert_allclose(mean.double().cpu().numpy(), s.mean(dim=1).cpu().numpy(),
                               rtol=2e-7, atol=0)


@pytest.mark.parametrize("own_stream", [False, True])
def test_bounded_wait_reports_timeout_and_recovers(own_stream):
    """The backward's finishers wait for one block more than exists, with a 2 ms limit: the
    wait runs out, the kernel returns, and ln_device_check reports LN_ETIMEOUT and re-zeroes
    the stream's workspace with work ordered on that stream.  Afterwards the same stream --
    the default one, or a non-blocking torch stream -- computes correct results again."""
    inp = synth.make_inputs(512, 768, "bf16", seed=9)
    L = ln.lib()
    st = torch.cuda.Stream() if own_stream else torch.cuda.current_stream()
    L.ln_debug_wait_test(2000)
    try:
        with torch.cuda.stream(st):
            d = P.to_device(inp)
            out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], EPS)
            if os.environ.get("LN_CHECK", "0") not in ("", "0"):
                # Check mode synchronises after every call, so the call itself reports it.
                with pytest.raises(ln.LnError) as e:
                    ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd)
                assert e.value.status == 5
            else:
                ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd)
                assert ln.device_check(st) == 5
    finally:
        L.ln_debug_wait_test(0)
    with torch.cuda.stream(st):
        assert ln.device_check(st) == 0
        gpu = P.run_gpu(inp, EPS)
    P.compare_all(gpu, P.run_oracle(inp, EPS), "bf16")


def test_launch_count_and_native_library_loaded():
    inp = synth.make_inputs(64, 768, "f32", seed=10)
    d = P.to_device(inp)
    out, res_out, mean, rstd = ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], EPS)
    assert ln.last_launch_count() == 1
    ln.bwd(d["dy"], res_out, d["gamma"], mean, rstd)
    assert ln.last_launch_count() == 1
    maps = open("/proc/self/maps").read()
    assert ln.LIB_PATH in maps


@pytest.mark.parametrize("name", ["bf16_8192x768", "bf16_4096x8192_mean100", "f32_64x768"])
def test_dependent_launches_in_a_cuda_graph(name):
    """Forward then backward on the forward's own outputs, chained on one stream and
    replayed from a CUDA graph: every kernel is launched with programmatic dependent launch
    and must wait for its predecessor before touching memory, so the graph replay gives
    bit for bit the results of the same calls run one at a time with a synchronisation in
    between."""
    w = synth.WORKLOADS[name]
    d = P.to_device(synth.workload_inputs(name, seed=5))
    ws = torch.zeros(ln.workspace_bytes(w.rows, w.cols), dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()

    def outputs():
        return dict(out=torch.full_like(d["x"], float("nan")),
                    res_out=torch.full_like(d["x"], float("nan")),
                    mean=torch.full((w.rows,), float("nan"), device="cuda"),
                    rstd=torch.full((w.rows,), float("nan"), device="cuda"),
                    dx=torch.full_like(d["x"], float("nan")),
                    dgamma=torch.full_like(d["gamma"], float("nan")),
                    dbeta=torch.full_like(d["gamma"], float("nan")))

    def chain(o, sync):
        ln.fwd(d["x"], d["res"], d["gamma"], d["beta"], w.eps, out=o["out"],
               res_out=o["res_out"], mean=o["mean"], rstd=o["rstd"], stream=st)
        if sync:
            st.synchronize()
        ln.bwd(d["dy"], o["res_out"], d["gamma"], o["mean"], o["rstd"], dx=o["dx"],
               dgamma=o["dgamma"], dbeta=o["dbeta"], workspace=ws, stream=st)
        if sync:
            st.synchronize()

    ref = outputs()
    chain(ref, sync=True)
    got = outputs()
    with torch.cuda.stream(st):
        chain(got, sync=False)  # warm-up outside the graph (plans, attributes)
    torch.cuda.synchronize()
    got = outputs()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        chain(got, sync=False)
    for _ in range(3):  # the same results every replay
        with torch.cuda.stream(st):
            g.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k].view(torch.uint8) if got[k].dtype != torch.float32
                               else got[k].view(torch.int32),
                               ref[k].view(torch.uint8) if ref[k].dtype != torch.float32
                               else ref[k].view(torch.int32)), k


@pytest.mark.parametrize("dtype,cols", [("bf16", 1280), ("bf16", 1024), ("f32", 1000), ("f32", 768)])
@pytest.mark.parametrize("rows", [2131, 4099])
def test_paired_rows_against_oracle(dtype, rows, cols):
    """Row counts that give blocks several 7-row tiles, an odd number of them and a partial
    last tile: the backward's warps take rows of consecutive tiles in pairs (bf16 rows of 4-5
    vectors per lane, fp32 rows) with an unpaired step at the end; every element is compared
    with the oracle."""
    inp = synth.make_inputs(rows, cols, dtype, seed=rows + cols)
    gpu = P.run_gpu(inp, EPS)
    ref = P.run_oracle(inp, EPS)
    P.compare_all(gpu, ref, dtype, conditioned=True)
