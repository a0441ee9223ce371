"""Float64 NumPy twin of the C oracle -- TEST INFRASTRUCTURE ONLY.

Vectorised, for small shapes.  It restates the same definitions as ``ln_oracle.c`` in
independent code so that the two can be compared:

* forward ("Accelerating Transformer on GPU (II): Training with LightSeq2", section 2.1;
  residual sum stored then normalised, "llm.c: the llmc/ CUDA kernel layer", section 3.2);
* backward, HW4 form, and dgamma/dbeta as column sums (same lecture, sections 2.1, 2.4);
* the fused residual-add + RMSNorm forward and backward ("GPU Performance from First
  Principles", section 6.1);
* the fused softmax forward ("Accelerating Transformer on GPU (I)", section 4.1) and backward
  ("... (II)", section 3.1);
* the fused cross-entropy with label smoothing ("... (I)", section 5.2), as -sum p log q;
* the bias + dropout + residual prologue ("... (I)", section 2.3) on Philox-4x32-10.
"""
from __future__ import annotations

import numpy as np

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(v):
    """Round float64 values to bf16 (8 significant bits, fp32 exponent range), ties to even."""
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    qexp = np.maximum(e - 8, -133)
    q = np.ldexp(np.ones_like(v), qexp)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.rint(v / q) * q
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, v), r)
    r = np.where((v == 0) | ~np.isfinite(v), v, r)
    return r


def round_io(v, io: str):
    v = np.asarray(v, dtype=np.float64)
    if io == "f32":
        return v.astype(np.float32).astype(np.float64)
    if io == "bf16":
        return round_bf16(v)
    return v


def ln_fwd(x, res, gamma, beta, eps: float, io: str = "f64"):
    x = np.asarray(x, dtype=np.float64)
    s = x if res is None else x + np.asarray(res, dtype=np.float64)
    s = round_io(s, io)
    mean = s.mean(axis=1)
    var = ((s - mean[:, None]) ** 2).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (s - mean[:, None]) * rstd[:, None]
    out = round_io(np.asarray(gamma, np.float64)[None, :] * xhat
                   + np.asarray(beta, np.float64)[None, :], io)
    return {"out": out, "res_out": s, "mean": mean, "rstd": rstd}


def ln_bwd(dy, xr, gamma, mean, rstd, io: str = "f64"):
    dy = np.asarray(dy, dtype=np.float64)
    xr = np.asarray(xr, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    mean = np.asarray(mean, dtype=np.float64)
    rstd = np.asarray(rstd, dtype=np.float64)
    m = dy.shape[1]
    xhat = (xr - mean[:, None]) * rstd[:, None]
    g = gamma[None, :] * dy
    sum_g = g.sum(axis=1, keepdims=True)
    sum_gx = (g * xhat).sum(axis=1, keepdims=True)
    dx = rstd[:, None] * (g - (sum_g + xhat * sum_gx) / m)
    dgamma = (dy * xhat).sum(axis=0)
    dbeta = dy.sum(axis=0)
    return {"dx": round_io(dx, io), "dgamma": round_io(dgamma, io), "dbeta": round_io(dbeta, io)}


def rms_fwd(x, res, gamma, eps: float, io: str = "f64"):
    """Fused residual-add + RMSNorm forward ("GPU Performance from First Principles", section
    6.1): s = x + res rounded to ``io``; out = gamma * s / sqrt(mean(s^2) + eps)."""
    x = np.asarray(x, dtype=np.float64)
    s = x if res is None else x + np.asarray(res, dtype=np.float64)
    s = round_io(s, io)
    rrms = 1.0 / np.sqrt((s * s).mean(axis=1) + eps)
    out = round_io(np.asarray(gamma, np.float64)[None, :] * (s * rrms[:, None]), io)
    return {"out": out, "res_out": s, "rrms": rrms}


def rms_bwd(dy, xr, gamma, rrms, io: str = "f64"):
    dy = np.asarray(dy, dtype=np.float64)
    xr = np.asarray(xr, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    rrms = np.asarray(rrms, dtype=np.float64)
    m = dy.shape[1]
    shat = xr * rrms[:, None]
    g = gamma[None, :] * dy
    dx = rrms[:, None] * (g - shat * (g * shat).sum(axis=1, keepdims=True) / m)
    dgamma = (dy * shat).sum(axis=0)
    return {"dx": round_io(dx, io), "dgamma": round_io(dgamma, io)}


def softmax_fwd(x, mask=None, scale: float = 1.0, io: str = "f64"):
    """Fused softmax forward ("Accelerating Transformer on GPU (I)", section 4.1)."""
    z = scale * np.asarray(x, dtype=np.float64)
    if mask is not None:
        mask = np.asarray(mask, dtype=np.float64)
        z = z + np.tile(mask, (-(-z.shape[0] // mask.shape[0]), 1))[: z.shape[0]]
    with np.errstate(invalid="ignore"):
        e = np.exp(z - z.max(axis=1, keepdims=True))
        return round_io(e / e.sum(axis=1, keepdims=True), io)


def softmax_bwd(dy, y, scale: float = 1.0, io: str = "f64"):
    """Fused softmax backward ("Accelerating Transformer on GPU (II)", section 3.1)."""
    dy = np.asarray(dy, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return round_io(scale * y * (dy - (dy * y).sum(axis=1, keepdims=True)), io)


def xent(x, targets, alpha: float = 0.0, dloss: float = 1.0, io: str = "f64"):
    """Fused cross-entropy with label smoothing ("Accelerating Transformer on GPU (I)",
    section 5.2), written as the page's sum: loss = -sum p log q, dx = dloss (q - p)."""
    x = np.asarray(x, dtype=np.float64)
    rows, V = x.shape
    t = np.asarray(targets)
    p = np.full((rows, V), alpha / V)
    p[np.arange(rows), t] += 1.0 - alpha
    z = x - x.max(axis=1, keepdims=True)
    logq = z - np.log(np.exp(z).sum(axis=1, keepdims=True))
    return {"loss": -(p * logq).sum(axis=1), "dx": round_io(dloss * (np.exp(logq) - p), io)}


_M0, _M1, _W0, _W1 = 0xD2511F53, 0xCD9E8D57, 0x9E3779B9, 0xBB67AE85


def philox4x32(c0, c1, c2, c3, k0, k1):
    """Philox-4x32-10 on uint64 arrays holding 32-bit words (vectorised over counters)."""
    m32 = np.uint64(0xFFFFFFFF)
    c = [np.asarray(v, dtype=np.uint64) for v in (c0, c1, c2, c3)]
    k = [np.uint64(k0), np.uint64(k1)]
    for r in range(10):
        if r:
            k = [(k[0] + np.uint64(_W0)) & m32, (k[1] + np.uint64(_W1)) & m32]
        p0 = np.uint64(_M0) * c[0]
        p1 = np.uint64(_M1) * c[2]
        c = [(p1 >> np.uint64(32)) ^ c[1] ^ k[0], p1 & m32, (p0 >> np.uint64(32)) ^ c[3] ^ k[1],
             p0 & m32]
    return c


def dropout_mask(seed, offset, p, rows, cols):
    i = np.arange(rows * cols, dtype=np.uint64)
    blk = i >> np.uint64(2)
    m32 = np.uint64(0xFFFFFFFF)
    w = philox4x32(blk & m32, blk >> np.uint64(32), np.full_like(blk, offset & 0xFFFFFFFF),
                   np.full_like(blk, offset >> 32), seed & 0xFFFFFFFF, seed >> 32)
    word = np.choose((i & np.uint64(3)).astype(np.int64), w)
    thr = min(int(np.floor(p * 2.0 ** 32)), 0xFFFFFFFF)
    return (word >= np.uint64(thr)).astype(np.uint8).reshape(rows, cols)


def bdr_ln_fwd(h, bias, res, gamma, beta, eps, p, seed, offset, io="f64"):
    h = np.asarray(h, dtype=np.float64)
    keep = dropout_mask(seed, offset, p, *h.shape)
    s = round_io(np.asarray(res, np.float64) + keep * (h + np.asarray(bias)[None, :]) / (1 - p), io)
    return ln_fwd(s, None, gamma, beta, eps, io)


def dropout_bwd(ds, p, seed, offset, io="f64"):
    ds = np.asarray(ds, dtype=np.float64)
    dh = dropout_mask(seed, offset, p, *ds.shape) * ds / (1 - p)
    return {"dh": round_io(dh, io), "dbias": round_io(dh.sum(axis=0), io)}
