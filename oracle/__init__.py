"""Float64 CPU oracle for fused residual-add + LayerNorm -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this package.  The CUDA library never calls it and shares no
code with it.

It covers the fused residual-add + LayerNorm (``ln_fwd``, ``ln_bwd``), the fused
residual-add + RMSNorm (``rms_fwd``, ``rms_bwd``), the fused softmax (``softmax_fwd``,
``softmax_bwd``), the fused cross-entropy (``xent``) and the bias + dropout + residual
prologue of the LayerNorm forward with its backward (``bdr_ln_fwd``, ``dropout_bwd``, on
a Philox-4x32-10 counter-based generator, ``philox4x32``).  Two independent implementations of the
same definitions live here:

* ``ln_oracle.c`` (float64 C, OpenMP over rows; built into ``libln_oracle.so`` by
  :func:`build`) -- the oracle proper, fast enough for the full-size configurations;
* ``numpy_ref.py`` (float64 NumPy, vectorised) -- a twin for small shapes, used to
  cross-check the C code.

Definitions followed (page titles and sections):

* forward: "Accelerating Transformer on GPU (II): Training with LightSeq2", section 2.1
  (xhat = (x - mu)/sigma, sigma = sqrt(var + eps), y = gamma*xhat + beta; mu and 1/sigma
  saved per row); biased variance as in "AI infra learning log (2): LayerNorm operator
  optimisation", section 2.1; residual sum written out first and normalised, as in
  "llm.c: the llmc/ CUDA kernel layer", section 3.2;
* backward: HW4 form and slides form of dx, dgamma = sum_rows dy*xhat, dbeta = sum_rows dy
  ("Training with LightSeq2", sections 2.1 and 2.4).

Every function here is pinned by tests marked ``not gpu`` (finite differences, torch float64
autograd, invariants, the pages' worked example, agreement of the two backward forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import numpy_ref  # noqa: F401  (re-exported for tests)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ln_oracle.c")
_LIB = os.path.join(_HERE, "libln_oracle.so")

IO_CODES = {"f64": 0, "f32": 1, "bf16": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ln_oracle.c`` with gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            d = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_ln_fwd.argtypes = [d, d, d, d, ctypes.c_double, i64, i64, ctypes.c_int,
                                          d, d, d, d, ctypes.c_int]
            lib.oracle_ln_fwd.restype = None
            lib.oracle_ln_bwd.argtypes = [d, d, d, d, d, i64, i64, ctypes.c_int, d, d, d,
                                          ctypes.c_int]
            lib.oracle_ln_bwd.restype = None
            lib.oracle_ln_bwd_dx_slides.argtypes = [d, d, d, d, d, i64, i64, d, ctypes.c_int]
            lib.oracle_ln_bwd_dx_slides.restype = None
            lib.oracle_rms_fwd.argtypes = [d, d, d, ctypes.c_double, i64, i64, ctypes.c_int,
                                           d, d, d, ctypes.c_int]
            lib.oracle_rms_fwd.restype = None
            lib.oracle_rms_bwd.argtypes = [d, d, d, d, i64, i64, ctypes.c_int, d, d,
                                           ctypes.c_int]
            lib.oracle_rms_bwd.restype = None
            lib.oracle_softmax_fwd.argtypes = [d, d, i64, ctypes.c_double, i64, i64,
                                               ctypes.c_int, d, ctypes.c_int]
            lib.oracle_softmax_fwd.restype = None
            lib.oracle_softmax_bwd.argtypes = [d, d, ctypes.c_double, i64, i64, ctypes.c_int, d,
                                               ctypes.c_int]
            lib.oracle_softmax_bwd.restype = None
            lib.oracle_xent.argtypes = [d, ctypes.POINTER(ctypes.c_int32), i64, i64,
                                        ctypes.c_double, ctypes.c_double, ctypes.c_int, d, d,
                                        ctypes.c_int]
            lib.oracle_xent.restype = None
            u32p = ctypes.POINTER(ctypes.c_uint32)
            u64 = ctypes.c_uint64
            lib.oracle_philox4x32.argtypes = [u32p, u32p, u32p]
            lib.oracle_philox4x32.restype = None
            lib.oracle_dropout_mask.argtypes = [u64, u64, ctypes.c_double, i64, i64,
                                                ctypes.POINTER(ctypes.c_uint8), ctypes.c_int]
            lib.oracle_dropout_mask.restype = None
            lib.oracle_bdr_ln_fwd.argtypes = [d, d, d, d, d, ctypes.c_double, ctypes.c_double,
                                              u64, u64, i64, i64, ctypes.c_int, d, d, d, d,
                                              ctypes.c_int]
            lib.oracle_bdr_ln_fwd.restype = None
            lib.oracle_dropout_bwd.argtypes = [d, ctypes.c_double, u64, u64, i64, i64,
                                               ctypes.c_int, d, d, ctypes.c_int]
            lib.oracle_dropout_bwd.restype = None
            lib.oracle_round_io.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.oracle_round_io.restype = ctypes.c_double
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def round_io(v, io: str):
    """Round float64 values to the I/O precision (round to nearest even)."""
    lib = _load()
    arr = _f64(v)
    flat = arr.reshape(-1)
    out = np.empty_like(flat)
    code = IO_CODES[io]
    for i in range(flat.size):
        out[i] = lib.oracle_round_io(float(flat[i]), code)
    return out.reshape(arr.shape)


def ln_fwd(x, res, gamma, beta, eps: float, io: str = "f64", threads: int = 0,
           want_out: bool = True, want_res_out: bool = True):
    """Forward of the fused residual-add + LayerNorm.

    ``x``, ``res``: [rows, cols] (``res`` may be None); ``gamma``, ``beta``: [cols].
    Returns a dict with ``out``, ``res_out`` (rounded to ``io``), ``mean`` and ``rstd``
    (float64, unrounded).
    """
    x = _f64(x)
    rows, cols = x.shape
    res = _f64(res)
    gamma = _f64(gamma)
    beta = _f64(beta)
    assert gamma.shape == (cols,) and beta.shape == (cols,)
    if res is not None:
        assert res.shape == x.shape
    out = np.empty((rows, cols)) if want_out else None
    res_out = np.empty((rows, cols)) if want_res_out else None
    mean = np.empty(rows)
    rstd = np.empty(rows)
    _load().oracle_ln_fwd(_ptr(x), _ptr(res), _ptr(gamma), _ptr(beta), float(eps), rows, cols,
                          IO_CODES[io], _ptr(out), _ptr(res_out), _ptr(mean), _ptr(rstd),
                          int(threads))
    return {"out": out, "res_out": res_out, "mean": mean, "rstd": rstd}


def ln_bwd(dy, xr, gamma, mean, rstd, io: str = "f64", threads: int = 0, want_dx: bool = True,
           want_dparams: bool = True):
    """Backward (HW4 form).  ``xr`` is the tensor the forward normalised (the stored residual
    sum when the forward had a residual, else x).  Returns ``dx`` [rows, cols] and
    ``dgamma``, ``dbeta`` [cols], rounded to ``io``."""
    dy = _f64(dy)
    rows, cols = dy.shape
    xr = _f64(xr)
    gamma = _f64(gamma)
    mean = _f64(mean)
    rstd = _f64(rstd)
    assert xr.shape == dy.shape and gamma.shape == (cols,)
    assert mean.shape == (rows,) and rstd.shape == (rows,)
    dx = np.empty((rows, cols)) if want_dx else None
    dgamma = np.empty(cols) if want_dparams else None
    dbeta = np.empty(cols) if want_dparams else None
    _load().oracle_ln_bwd(_ptr(dy), _ptr(xr), _ptr(gamma), _ptr(mean), _ptr(rstd), rows, cols,
                          IO_CODES[io], _ptr(dx), _ptr(dgamma), _ptr(dbeta), int(threads))
    return {"dx": dx, "dgamma": dgamma, "dbeta": dbeta}


def ln_bwd_dx_slides(dy, xr, gamma, mean, rstd, threads: int = 0):
    """dx by the slides form (raw x in the second sum), float64, unrounded."""
    dy = _f64(dy)
    rows, cols = dy.shape
    xr = _f64(xr)
    gamma = _f64(gamma)
    mean = _f64(mean)
    rstd = _f64(rstd)
    dx = np.empty((rows, cols))
    _load().oracle_ln_bwd_dx_slides(_ptr(dy), _ptr(xr), _ptr(gamma), _ptr(mean), _ptr(rstd),
                                    rows, cols, _ptr(dx), int(threads))
    return dx


def rms_fwd(x, res, gamma, eps: float, io: str = "f64", threads: int = 0, want_out: bool = True,
            want_res_out: bool = True):
    """Forward of the fused residual-add + RMSNorm ("GPU Performance from First Principles",
    section 6.1): s = x + res (rounded to ``io``), r = 1/sqrt(mean(s^2) + eps),
    out = gamma * s * r.  Returns ``out``, ``res_out`` (rounded to ``io``) and ``rrms`` (r,
    float64, unrounded)."""
    x = _f64(x)
    rows, cols = x.shape
    res = _f64(res)
    gamma = _f64(gamma)
    assert gamma.shape == (cols,)
    if res is not None:
        assert res.shape == x.shape
    out = np.empty((rows, cols)) if want_out else None
    res_out = np.empty((rows, cols)) if want_res_out else None
    rrms = np.empty(rows)
    _load().oracle_rms_fwd(_ptr(x), _ptr(res), _ptr(gamma), float(eps), rows, cols,
                           IO_CODES[io], _ptr(out), _ptr(res_out), _ptr(rrms), int(threads))
    return {"out": out, "res_out": res_out, "rrms": rrms}


def rms_bwd(dy, xr, gamma, rrms, io: str = "f64", threads: int = 0, want_dx: bool = True,
            want_dgamma: bool = True):
    """Backward of the fused residual-add + RMSNorm: ``dx`` = r (g - shat sum(g shat)/m) with
    shat = xr * r, g = gamma * dy, and ``dgamma`` = sum over rows of dy * shat, rounded to
    ``io``.  ``xr`` is the tensor the forward normalised."""
    dy = _f64(dy)
    rows, cols = dy.shape
    xr = _f64(xr)
    gamma = _f64(gamma)
    rrms = _f64(rrms)
    assert xr.shape == dy.shape and gamma.shape == (cols,) and rrms.shape == (rows,)
    dx = np.empty((rows, cols)) if want_dx else None
    dgamma = np.empty(cols) if want_dgamma else None
    _load().oracle_rms_bwd(_ptr(dy), _ptr(xr), _ptr(gamma), _ptr(rrms), rows, cols,
                           IO_CODES[io], _ptr(dx), _ptr(dgamma), int(threads))
    return {"dx": dx, "dgamma": dgamma}


def softmax_fwd(x, mask=None, scale: float = 1.0, io: str = "f64", threads: int = 0):
    """Fused softmax forward ("Accelerating Transformer on GPU (I)", section 4.1): per row,
    y = softmax(scale * x + mask), the additive mask's rows repeating every mask.shape[0]
    rows.  Returns y rounded to ``io``."""
    x = _f64(x)
    rows, cols = x.shape
    mask = _f64(mask)
    mask_rows = 1
    if mask is not None:
        assert mask.ndim == 2 and mask.shape[1] == cols
        mask_rows = mask.shape[0]
    y = np.empty((rows, cols))
    _load().oracle_softmax_fwd(_ptr(x), _ptr(mask), mask_rows, float(scale), rows, cols,
                               IO_CODES[io], _ptr(y), int(threads))
    return y


def softmax_bwd(dy, y, scale: float = 1.0, io: str = "f64", threads: int = 0):
    """Fused softmax backward ("Accelerating Transformer on GPU (II)", section 3.1):
    dx = scale * y * (dy - sum(dy * y)), rounded to ``io``."""
    dy = _f64(dy)
    rows, cols = dy.shape
    y = _f64(y)
    assert y.shape == dy.shape
    dx = np.empty((rows, cols))
    _load().oracle_softmax_bwd(_ptr(dy), _ptr(y), float(scale), rows, cols, IO_CODES[io],
                               _ptr(dx), int(threads))
    return dx


def xent(x, targets, alpha: float = 0.0, dloss: float = 1.0, io: str = "f64", threads: int = 0,
         want_dx: bool = True):
    """Fused cross-entropy with label smoothing ("Accelerating Transformer on GPU (I)",
    section 5.2): per row, loss = log Z + m - [(1 - alpha) x_t + (alpha / V) sum x] and
    dx = dloss * (softmax(x) - p), p = (1 - alpha) onehot(t) + alpha / V.  Returns
    ``losses`` (float64) and ``dx`` (rounded to ``io``)."""
    x = _f64(x)
    rows, V = x.shape
    t = np.ascontiguousarray(np.asarray(targets, dtype=np.int32))
    assert t.shape == (rows,) and np.all((t >= 0) & (t < V))
    losses = np.empty(rows)
    dx = np.empty((rows, V)) if want_dx else None
    _load().oracle_xent(_ptr(x), t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), rows, V,
                        float(alpha), float(dloss), IO_CODES[io], _ptr(losses), _ptr(dx),
                        int(threads))
    return {"loss": losses, "dx": dx}


def philox4x32(ctr, key):
    """Philox-4x32-10 of one counter (4 words) under one key (2 words): 4 words."""
    c = (ctypes.c_uint32 * 4)(*ctr)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    _load().oracle_philox4x32(c, k, o)
    return list(o)


def dropout_mask(seed: int, offset: int, p: float, rows: int, cols: int, threads: int = 0):
    """uint8 [rows, cols]: 1 where the element is kept (see oracle_dropout_mask)."""
    keep = np.empty((rows, cols), dtype=np.uint8)
    _load().oracle_dropout_mask(seed, offset, float(p), rows, cols,
                                keep.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                int(threads))
    return keep


def bdr_ln_fwd(h, bias, res, gamma, beta, eps: float, p: float, seed: int, offset: int,
               io: str = "f64", threads: int = 0):
    """Bias + dropout + residual prologue ("Accelerating Transformer on GPU (I)", section
    2.3) fused with the LayerNorm forward: s = res + keep * (h + bias) / (1 - p), rounded to
    ``io``, then LN(s).  Returns ``out``, ``res_out``, ``mean``, ``rstd``."""
    h = _f64(h)
    rows, cols = h.shape
    res = _f64(res)
    out = np.empty((rows, cols))
    res_out = np.empty((rows, cols))
    mean = np.empty(rows)
    rstd = np.empty(rows)
    _load().oracle_bdr_ln_fwd(_ptr(h), _ptr(_f64(bias)), _ptr(res), _ptr(_f64(gamma)),
                              _ptr(_f64(beta)), float(eps), float(p), seed, offset, rows, cols,
                              IO_CODES[io], _ptr(out), _ptr(res_out), _ptr(mean), _ptr(rstd),
                              int(threads))
    return {"out": out, "res_out": res_out, "mean": mean, "rstd": rstd}


def dropout_bwd(ds, p: float, seed: int, offset: int, io: str = "f64", threads: int = 0):
    """Backward of the prologue: dh = ds * keep / (1 - p), dbias = sum over rows of dh."""
    ds = _f64(ds)
    rows, cols = ds.shape
    dh = np.empty((rows, cols))
    dbias = np.empty(cols)
    _load().oracle_dropout_bwd(_ptr(ds), float(p), seed, offset, rows, cols, IO_CODES[io],
                               _ptr(dh), _ptr(dbias), int(threads))
    return {"dh": dh, "dbias": dbias}
