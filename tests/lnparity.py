"""Helpers for the GPU parity tests: run the CUDA path through the binding (C ABI) and the
float64 oracle on the same seeded inputs, and compare them element by element.

Tolerances (the ones the tests assert):

* fp32 I/O: out, res_out and dx within 2e-5 absolute, or 4 fp32 ulps of the oracle value
  where that is larger (|value| >= 64: at 256 the fp32 spacing alone is 3e-5, so no fp32
  computation of more than one rounding can promise 2e-5 there; dx of a constant row is
  rstd * (g - mean g) with rstd = eps^-1/2 ~ 316, hundreds in size); mean, rstd, dgamma and
  dbeta within 2e-5 * max(1, |oracle|) (column sums over 262144 rows reach ~1e3, where the
  fp32 spacing alone is ~1e-4, so a fixed 2e-5 absolute bound would ask for more than fp32
  can hold).
* bf16 I/O: every bf16 output within 2 bf16 ulps of the oracle value, the ulp taken at
  max(|oracle|, 2^-14) (a plain "2 ulps of the value" cannot be met for values that round
  to almost 0 after an fp32 computation: the fp32 arithmetic itself is ~1e-7 absolute);
  res_out bit-exact (it is one correctly rounded addition); mean and rstd (fp32) as above.

Conditioning term (edge-case sweeps only, never the five workloads): the backward receives
mu stored in fp32.  A stored mean off by dmu moves xhat by rstd*dmu, dx by up to
rstd^2 * dmu * (|sum g xhat| + |xhat_j| |sum g|) / n and dgamma_j by sum_rows |dy| rstd dmu
(first order).  With dmu = 2^-22 (|mu| + max|s - mu|) this is below 1e-9 for rows whose
spread is not tiny next to their mean and eps, but rows of two or three nearly equal values
(var << eps, rstd ~ 300) can reach 1e-2: no fp32-stats backward can do better there.  The
sweep adds twice this term (and 2^-21 |dx| for the fp32 rounding of rstd) to the bound.

Column-sum term (every comparison of dgamma and dbeta): each term dy * xhat of a column
sum reaches the sum through a few fp32 roundings (xhat from the fp32-stored mean and rstd,
the product, the accumulation), independent from row to row.  Their sum over n rows is a
sum of n independent, zero-mean errors |e_r| <= k u |t_r| (u = 2^-24, k <= 6), so by
Hoeffding's inequality |sum e_r| <= 6 k u ||t||_2 except with probability 2 exp(-18)
(about 3e-8 per column).  A column whose terms cancel to almost 0 cannot meet "2e-5" or
"2 ulps of the value" in fp32 once n is large (262144 rows: ||t||_2 ~ 400, and the bare
rounding of the stored rstd alone moves the sum by ~1e-5), so this allowance, 36 u ||t||_2,
is added to the stated bound for dgamma (t = dy * xhat) and dbeta (t = dy).  Every
comparison also counts how many elements exceed the bare stated bound (``n_over_stated``).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import layernorm_ln_fwd_gb300 as ln
import oracle

BF16_FLOOR = 2.0 ** -14
F32_ABS = 2e-5

_REPORT = os.environ.get("LN_PARITY_REPORT")


def report(info: dict) -> None:
    """Append one comparison summary as a JSON line to $LN_PARITY_REPORT, if set."""
    if not _REPORT:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    with open(_REPORT, "a") as f:
        f.write(json.dumps(dict(info, test=test)) + "\n")


def to64(t) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def ulp_bf16(v) -> np.ndarray:
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), BF16_FLOOR)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def io_of(dtype) -> str:
    return {torch.float32: "f32", torch.bfloat16: "bf16"}[dtype]


def ulp_f32(v) -> np.ndarray:
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 23)


def tolerance(name: str, ref: np.ndarray, io: str) -> np.ndarray:
    if name in ("mean", "rstd", "rrms", "loss") or (io == "f32" and name in ("dgamma", "dbeta")):
        return F32_ABS * np.maximum(1.0, np.abs(ref))
    if io == "f32":
        # 2e-5 absolute; from |value| >= 64 on, where fp32 values are more than 5e-6 apart,
        # 4 fp32 ulps of the oracle value (a few roundings of a value that size).
        return np.maximum(F32_ABS, 4.0 * ulp_f32(ref))
    return 2.0 * ulp_bf16(ref)


def compare(name: str, gpu: np.ndarray, ref: np.ndarray, io: str, extra=None) -> dict:
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    base = tolerance(name, ref, io)
    tol = base if extra is None else base + extra
    bad = ~(err <= tol)  # NaN counts as bad
    worst = int(np.argmax(err / tol)) if err.size else 0
    info = {"name": name, "io": io, "n": int(err.size),
            "max_abs": float(err.max()) if err.size else 0.0,
            "worst_ratio": float((err / tol).max()) if err.size else 0.0,
            "n_over_stated": int((~(err <= base)).sum()), "n_bad": int(bad.sum())}
    report(info)
    if bad.any():
        idx = np.unravel_index(worst, err.shape)
        raise AssertionError(
            f"{name}: {info['n_bad']} of {err.size} outside tolerance; worst at {idx}: gpu "
            f"{gpu[idx]!r} oracle {ref[idx]!r} tol {tol[idx]!r}")
    return info


def to_device(inp: dict, dev="cuda") -> dict:
    return {k: v.to(dev) for k, v in inp.items()}


def run_gpu(inp: dict, eps: float, has_res: bool = True, write_res: bool = True,
            workspace=None) -> dict:
    d = to_device(inp)
    res = d["res"] if has_res else None
    out, res_out, mean, rstd = ln.fwd(d["x"], res, d["gamma"], d["beta"], eps,
                                      write_res_out=write_res)
    r = {"out": out, "mean": mean, "rstd": rstd}
    if res_out is not None:
        r["res_out"] = res_out
    if has_res and res_out is None:  # nothing to feed the backward: forward only
        torch.cuda.synchronize()
        return r
    xr = res_out if has_res else d["x"]
    r["dx"], r["dgamma"], r["dbeta"] = ln.bwd(d["dy"], xr, d["gamma"], mean, rstd,
                                              workspace=workspace)
    torch.cuda.synchronize()
    return r


def conditioning(f: dict, dy: np.ndarray, gamma: np.ndarray, dx: np.ndarray) -> dict:
    """Twice the first-order effect of storing mu in fp32 (see the module docstring)."""
    s, mu, rs = f["res_out"], f["mean"], f["rstd"]
    n = s.shape[1]
    xhat = (s - mu[:, None]) * rs[:, None]
    g = gamma[None, :] * dy
    sg = g.sum(axis=1, keepdims=True)
    sgx = (g * xhat).sum(axis=1, keepdims=True)
    dmu = 2.0 ** -22 * (np.abs(mu) + np.abs(s - mu[:, None]).max(axis=1))
    e_dx = 2 * (rs ** 2 * dmu)[:, None] * (np.abs(sgx) + np.abs(xhat) * np.abs(sg)) / n
    e_dx += 2.0 ** -21 * np.abs(dx)
    e_dg = 2 * (np.abs(dy) * (rs * dmu)[:, None]).sum(axis=0)
    return {"dx": e_dx, "dgamma": e_dg}


def colsum_allowance(dy: np.ndarray, xhat: np.ndarray) -> dict:
    """36 * 2^-24 * ||terms||_2 for the column sums dgamma and dbeta (module docstring)."""
    k = 36.0 * 2.0 ** -24
    return {"dgamma": k * np.sqrt(((dy * xhat) ** 2).sum(axis=0)),
            "dbeta": k * np.sqrt((dy ** 2).sum(axis=0))}


def run_oracle(inp: dict, eps: float, has_res: bool = True, rows_idx=None,
               want_dparams: bool = True) -> dict:
    io = io_of(inp["x"].dtype)
    sel = (lambda t: t) if rows_idx is None else (lambda t: t[rows_idx])
    x = to64(sel(inp["x"]))
    res = to64(sel(inp["res"])) if has_res else None
    dy = to64(sel(inp["dy"]))
    gamma = to64(inp["gamma"])
    beta = to64(inp["beta"])
    f = oracle.ln_fwd(x, res, gamma, beta, eps, io=io)
    b = oracle.ln_bwd(dy, f["res_out"], gamma, f["mean"], f["rstd"], io=io,
                      want_dparams=want_dparams and rows_idx is None)
    r = {"out": f["out"], "res_out": f["res_out"], "mean": f["mean"], "rstd": f["rstd"],
         "dx": b["dx"]}
    if want_dparams and rows_idx is None:
        r["dgamma"], r["dbeta"] = b["dgamma"], b["dbeta"]
    r["_conditioning"] = conditioning(f, dy, gamma, b["dx"])
    xhat = (f["res_out"] - f["mean"][:, None]) * f["rstd"][:, None]
    r["_colsum"] = colsum_allowance(dy, xhat)
    return r


def oracle_dparams(inp: dict, eps: float, has_res: bool = True) -> dict:
    """dgamma and dbeta over all rows (the forward is needed for mean, rstd, res_out)."""
    io = io_of(inp["x"].dtype)
    x = to64(inp["x"])
    res = to64(inp["res"]) if has_res else None
    f = oracle.ln_fwd(x, res, to64(inp["gamma"]), to64(inp["beta"]), eps, io=io,
                      want_out=False)
    del x, res
    dy = to64(inp["dy"])
    b = oracle.ln_bwd(dy, f["res_out"], to64(inp["gamma"]), f["mean"], f["rstd"], io=io,
                      want_dx=False)
    xhat = (f["res_out"] - f["mean"][:, None]) * f["rstd"][:, None]
    return {"dgamma": b["dgamma"], "dbeta": b["dbeta"], "_colsum": colsum_allowance(dy, xhat)}


def compare_all(gpu: dict, ref: dict, io: str, rows_idx=None, conditioned: bool = False) -> list:
    """Compare every output; ``conditioned`` adds the fp32-mean conditioning term."""
    infos = []
    cond = ref.get("_conditioning", {}) if conditioned else {}
    colsum = ref.get("_colsum", {})
    for name, r in ref.items():
        if name not in gpu or name.startswith("_"):
            continue
        g = gpu[name]
        if rows_idx is not None and name not in ("dgamma", "dbeta"):
            g = g[torch.as_tensor(rows_idx, device=g.device)]
        extra = None
        for part in (cond.get(name), colsum.get(name)):
            if part is not None:
                extra = part if extra is None else extra + part
        infos.append(compare(name, to64(g), r, io, extra=extra))
    if "res_out" in gpu and "res_out" in ref and io == "bf16":
        g = gpu["res_out"] if rows_idx is None else gpu["res_out"][
            torch.as_tensor(rows_idx, device=gpu["res_out"].device)]
        np.testing.assert_array_equal(to64(g), ref["res_out"])
    return infos


def stored_stats_inputs(inp: dict, eps: float) -> dict:
    """Backward inputs as the forward stores them, taken from the ORACLE's forward: res_out
    (already in the I/O type) and mean, rstd rounded to fp32 (the API's storage type)."""
    io = io_of(inp["x"].dtype)
    f = oracle.ln_fwd(to64(inp["x"]), to64(inp["res"]), to64(inp["gamma"]), to64(inp["beta"]),
                      eps, io=io, want_out=False)
    return {"res_out": f["res_out"], "mean": oracle.round_io(f["mean"], "f32"),
            "rstd": oracle.round_io(f["rstd"], "f32")}
