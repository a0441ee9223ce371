"""GB300 (sm_103a) fused residual-add + LayerNorm (and RMSNorm), forward and backward.

A thin ctypes binding over the C ABI of ``libln.so`` (declared in ``include/ln.h``).  It only
marshals arguments: it checks dtypes, shapes, devices and contiguity, allocates outputs with
torch when the caller does not pass them, and hands raw device pointers and the current
CUDA stream to the library.  Every step of the computation runs in the library's kernels;
there is no fallback: if ``libln.so`` is missing, the first call raises RuntimeError.

Forward (``fwd``): s = x + res is written as ``res_out``; out = gamma * (s - mu) * rstd + beta,
with per-row fp32 ``mean`` and ``rstd``.  Backward (``bwd``): dx with respect to s (hence to
both x and res), dgamma and dbeta, the latter bitwise reproducible.  ``rms_fwd`` and
``rms_bwd`` do the same for the fused residual-add + RMSNorm ("GPU Performance from First
Principles", section 6.1).  Definitions:
"Accelerating Transformer on GPU (II): Training with LightSeq2", sections 2.1, 2.2 and 2.4;
residual fusion as in "llm.c: the llmc/ CUDA kernel layer", section 3.2.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libln.so")

STATUS = {0: "LN_OK", 1: "LN_EINVAL", 2: "LN_EALIGN", 3: "LN_EUNSUPPORTED", 4: "LN_ECUDA",
          5: "LN_ETIMEOUT", 6: "LN_ENOSPACE"}
MAX_COLS = 16384
PATH_AUTO, PATH_WARP, PATH_BLOCK, PATH_SCALAR = 0, 1, 2, 3

# Every symbol include/ln.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_INT = ctypes.c_int
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64
SIGNATURES = {
    "ln_fwd_f32": (_INT, [_P, _P, _P, _P, _F, _I64, _I64, _P, _P, _P, _P, _P]),
    "ln_fwd_bf16": (_INT, [_P, _P, _P, _P, _F, _I64, _I64, _P, _P, _P, _P, _P]),
    "ln_bwd_f32": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "ln_bwd_bf16": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "ln_bwd_workspace_bytes": (_SZ, [_I64, _I64]),
    "ln_bwd_f32_ws": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "ln_bwd_bf16_ws": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "ln_device_check": (_INT, [_P]),
    "ln_release": (_INT, []),
    "ln_status_str": (ctypes.c_char_p, [_INT]),
    "ln_last_cuda_error": (_INT, []),
    "ln_version": (_INT, []),
    "ln_debug_force_path": (_INT, [_INT]),
    "ln_debug_wait_test": (None, [ctypes.c_uint]),
    "ln_last_launch_count": (_INT, []),
    "ln_bwd_bf16_noalloc": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "ln_rms_fwd_f32": (_INT, [_P, _P, _P, _F, _I64, _I64, _P, _P, _P, _P]),
    "ln_rms_fwd_bf16": (_INT, [_P, _P, _P, _F, _I64, _I64, _P, _P, _P, _P]),
    "ln_rms_bwd_f32": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "ln_rms_bwd_bf16": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "ln_rms_bwd_f32_ws": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "ln_rms_bwd_bf16_ws": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "ln_softmax_fwd_f32": (_INT, [_P, _P, _I64, _F, _I64, _I64, _P, _P]),
    "ln_softmax_fwd_bf16": (_INT, [_P, _P, _I64, _F, _I64, _I64, _P, _P]),
    "ln_softmax_bwd_f32": (_INT, [_P, _P, _F, _I64, _I64, _P, _P]),
    "ln_softmax_bwd_bf16": (_INT, [_P, _P, _F, _I64, _I64, _P, _P]),
    "ln_xent_f32": (_INT, [_P, _P, _I64, _I64, _F, _F, _P, _P, _P]),
    "ln_xent_bf16": (_INT, [_P, _P, _I64, _I64, _F, _F, _P, _P, _P]),
    "ln_fwd_bias_dropout_f32": (_INT, [_P, _P, _P, _P, _P, _F, _F, _U64, _U64, _I64, _I64, _P, _P,
                                       _P, _P, _P]),
    "ln_fwd_bias_dropout_bf16": (_INT, [_P, _P, _P, _P, _P, _F, _F, _U64, _U64, _I64, _I64, _P,
                                        _P, _P, _P, _P]),
    "ln_dropout_bwd_f32": (_INT, [_P, _F, _U64, _U64, _I64, _I64, _P, _P, _P]),
    "ln_dropout_bwd_bf16": (_INT, [_P, _F, _U64, _U64, _I64, _I64, _P, _P, _P]),
    "ln_dropout_bwd_f32_ws": (_INT, [_P, _F, _U64, _U64, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "ln_dropout_bwd_bf16_ws": (_INT, [_P, _F, _U64, _U64, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "ln_dropout_keep_bytes": (_SZ, [_I64, _I64]),
    "ln_fwd_bias_dropout_keep_f32": (_INT, [_P, _P, _P, _P, _P, _F, _F, _U64, _U64, _I64, _I64,
                                            _P, _P, _P, _P, _P, _P]),
    "ln_fwd_bias_dropout_keep_bf16": (_INT, [_P, _P, _P, _P, _P, _F, _F, _U64, _U64, _I64, _I64,
                                             _P, _P, _P, _P, _P, _P]),
    "ln_dropout_bwd_keep_f32": (_INT, [_P, _F, _P, _I64, _I64, _P, _P, _P]),
    "ln_dropout_bwd_keep_bf16": (_INT, [_P, _F, _P, _I64, _I64, _P, _P, _P]),
    "ln_dropout_bwd_keep_f32_ws": (_INT, [_P, _F, _P, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "ln_dropout_bwd_keep_bf16_ws": (_INT, [_P, _F, _P, _I64, _I64, _P, _P, _P, _SZ, _P]),
}


class LnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = STATUS.get(status, str(status))
        if status == 4 and _lib is not None:
            msg += f" (cudaError {_lib.ln_last_cuda_error()})"
        super().__init__(f"{fn} returned {msg}")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded ``libln.so`` with argument types set.  Raises RuntimeError if missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m layernorm_ln_fwd_gb300.build`")
            cdll = ctypes.CDLL(LIB_PATH)
            for name, (restype, argtypes) in SIGNATURES.items():
                fn = getattr(cdll, name)
                fn.restype = restype
                fn.argtypes = argtypes
            _lib = cdll
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise LnError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _suffix(dtype) -> str:
    import torch
    if dtype == torch.float32:
        return "f32"
    if dtype == torch.bfloat16:
        return "bf16"
    raise TypeError(f"unsupported dtype {dtype}: use torch.float32 or torch.bfloat16")


def _need(t, name, shape, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def fwd(x, res, gamma, beta, eps: float = 1e-5, out=None, res_out=None, mean=None, rstd=None,
        write_res_out: bool = True, stream=None):
    """Forward.  x, res: [rows, cols] (res may be None); gamma, beta: [cols].

    Returns (out, res_out, mean, rstd); res_out is None when ``write_res_out`` is False and
    no ``res_out`` tensor is given.
    """
    import torch
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    rows, cols = x.shape
    dt, dev = x.dtype, x.device
    sfx = _suffix(dt)
    _need(x, "x", (rows, cols), dt, dev)
    if res is not None:
        _need(res, "res", (rows, cols), dt, dev)
    _need(gamma, "gamma", (cols,), dt, dev)
    _need(beta, "beta", (cols,), dt, dev)
    out = torch.empty_like(x) if out is None else _need(out, "out", (rows, cols), dt, dev)
    if res_out is None and write_res_out:
        res_out = torch.empty_like(x)
    elif res_out is not None:
        _need(res_out, "res_out", (rows, cols), dt, dev)
    mean = (torch.empty(rows, dtype=torch.float32, device=dev) if mean is None
            else _need(mean, "mean", (rows,), torch.float32, dev))
    rstd = (torch.empty(rows, dtype=torch.float32, device=dev) if rstd is None
            else _need(rstd, "rstd", (rows,), torch.float32, dev))
    name = f"ln_fwd_{sfx}"
    _check(name, getattr(lib(), name)(_ptr(x), _ptr(res), _ptr(gamma), _ptr(beta), float(eps),
                                      rows, cols, _ptr(out), _ptr(res_out), _ptr(mean),
                                      _ptr(rstd), _stream(stream)))
    return out, res_out, mean, rstd


def bwd(dy, x_or_res_out, gamma, mean, rstd, dx=None, dgamma=None, dbeta=None, workspace=None,
        stream=None):
    """Backward.  Returns (dx, dgamma, dbeta).

    ``workspace``: an optional caller-owned uint8 CUDA tensor of at least
    ``workspace_bytes(rows, cols)`` bytes, zeroed before its first use (selects the _ws
    entry point); by default the library's own per-stream workspace is used.
    """
    import torch
    if dy.dim() != 2:
        raise ValueError("dy must be 2-D [rows, cols]")
    rows, cols = dy.shape
    dt, dev = dy.dtype, dy.device
    sfx = _suffix(dt)
    _need(dy, "dy", (rows, cols), dt, dev)
    _need(x_or_res_out, "x_or_res_out", (rows, cols), dt, dev)
    _need(gamma, "gamma", (cols,), dt, dev)
    _need(mean, "mean", (rows,), torch.float32, dev)
    _need(rstd, "rstd", (rows,), torch.float32, dev)
    dx = torch.empty_like(dy) if dx is None else _need(dx, "dx", (rows, cols), dt, dev)
    dgamma = (torch.empty(cols, dtype=dt, device=dev) if dgamma is None
              else _need(dgamma, "dgamma", (cols,), dt, dev))
    dbeta = (torch.empty(cols, dtype=dt, device=dev) if dbeta is None
             else _need(dbeta, "dbeta", (cols,), dt, dev))
    args = [_ptr(dy), _ptr(x_or_res_out), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dx),
            _ptr(dgamma), _ptr(dbeta), rows, cols]
    if workspace is None:
        name = f"ln_bwd_{sfx}"
        _check(name, getattr(lib(), name)(*args, _stream(stream)))
    else:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the same device")
        nbytes = workspace.numel() * workspace.element_size()
        name = f"ln_bwd_{sfx}_ws"
        _check(name, getattr(lib(), name)(*args, _ptr(workspace), nbytes, _stream(stream)))
    return dx, dgamma, dbeta


def workspace_bytes(rows: int, cols: int) -> int:
    """Bytes of caller-owned workspace the backward needs on the current device."""
    return int(lib().ln_bwd_workspace_bytes(rows, cols))


def device_check(stream=None) -> int:
    """Synchronize ``stream`` and return the device status (0 = LN_OK, 5 = LN_ETIMEOUT)."""
    return int(lib().ln_device_check(_stream(stream)))


def release() -> None:
    _check("ln_release", lib().ln_release())


def force_path(path: int) -> int:
    """Select a kernel family for later calls (0 auto, 1 warp, 2 block, 3 scalar)."""
    return int(lib().ln_debug_force_path(path))


def last_launch_count() -> int:
    return int(lib().ln_last_launch_count())


def rms_fwd(x, res, gamma, eps: float = 1e-5, out=None, res_out=None, rrms=None,
            write_res_out: bool = True, stream=None):
    """Fused residual-add + RMSNorm forward.  x, res: [rows, cols] (res may be None); gamma:
    [cols].  Returns (out, res_out, rrms): out = gamma * s * rrms, s = x + res stored as
    res_out, rrms = 1 / sqrt(mean(s^2) + eps) per row (fp32)."""
    import torch
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    rows, cols = x.shape
    dt, dev = x.dtype, x.device
    sfx = _suffix(dt)
    _need(x, "x", (rows, cols), dt, dev)
    if res is not None:
        _need(res, "res", (rows, cols), dt, dev)
    _need(gamma, "gamma", (cols,), dt, dev)
    out = torch.empty_like(x) if out is None else _need(out, "out", (rows, cols), dt, dev)
    if res_out is None and write_res_out:
        res_out = torch.empty_like(x)
    elif res_out is not None:
        _need(res_out, "res_out", (rows, cols), dt, dev)
    rrms = (torch.empty(rows, dtype=torch.float32, device=dev) if rrms is None
            else _need(rrms, "rrms", (rows,), torch.float32, dev))
    name = f"ln_rms_fwd_{sfx}"
    _check(name, getattr(lib(), name)(_ptr(x), _ptr(res), _ptr(gamma), float(eps), rows, cols,
                                      _ptr(out), _ptr(res_out), _ptr(rrms), _stream(stream)))
    return out, res_out, rrms


def rms_bwd(dy, x_or_res_out, gamma, rrms, dx=None, dgamma=None, workspace=None, stream=None):
    """Fused residual-add + RMSNorm backward.  Returns (dx, dgamma); ``workspace`` as for
    :func:`bwd`."""
    import torch
    if dy.dim() != 2:
        raise ValueError("dy must be 2-D [rows, cols]")
    rows, cols = dy.shape
    dt, dev = dy.dtype, dy.device
    sfx = _suffix(dt)
    _need(dy, "dy", (rows, cols), dt, dev)
    _need(x_or_res_out, "x_or_res_out", (rows, cols), dt, dev)
    _need(gamma, "gamma", (cols,), dt, dev)
    _need(rrms, "rrms", (rows,), torch.float32, dev)
    dx = torch.empty_like(dy) if dx is None else _need(dx, "dx", (rows, cols), dt, dev)
    dgamma = (torch.empty(cols, dtype=dt, device=dev) if dgamma is None
              else _need(dgamma, "dgamma", (cols,), dt, dev))
    args = [_ptr(dy), _ptr(x_or_res_out), _ptr(gamma), _ptr(rrms), _ptr(dx), _ptr(dgamma),
            rows, cols]
    if workspace is None:
        name = f"ln_rms_bwd_{sfx}"
        _check(name, getattr(lib(), name)(*args, _stream(stream)))
    else:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the same device")
        nbytes = workspace.numel() * workspace.element_size()
        name = f"ln_rms_bwd_{sfx}_ws"
        _check(name, getattr(lib(), name)(*args, _ptr(workspace), nbytes, _stream(stream)))
    return dx, dgamma


def softmax_fwd(x, mask=None, scale: float = 1.0, y=None, stream=None):
    """Fused row softmax: y = softmax(scale * x + mask[r % mask_rows]) per row r.  x:
    [rows, cols]; mask: None or [mask_rows, cols] (additive, -inf removes an entry)."""
    import torch
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    rows, cols = x.shape
    dt, dev = x.dtype, x.device
    sfx = _suffix(dt)
    _need(x, "x", (rows, cols), dt, dev)
    mask_rows = 1
    if mask is not None:
        if mask.dim() != 2:
            raise ValueError("mask must be 2-D [mask_rows, cols]")
        mask_rows = mask.shape[0]
        _need(mask, "mask", (mask_rows, cols), dt, dev)
    y = torch.empty_like(x) if y is None else _need(y, "y", (rows, cols), dt, dev)
    name = f"ln_softmax_fwd_{sfx}"
    _check(name, getattr(lib(), name)(_ptr(x), _ptr(mask), mask_rows, float(scale), rows, cols,
                                      _ptr(y), _stream(stream)))
    return y


def softmax_bwd(dy, y, scale: float = 1.0, dx=None, stream=None):
    """Fused row softmax backward: dx = scale * y * (dy - sum(dy * y)) per row."""
    import torch
    if dy.dim() != 2:
        raise ValueError("dy must be 2-D [rows, cols]")
    rows, cols = dy.shape
    dt, dev = dy.dtype, dy.device
    sfx = _suffix(dt)
    _need(dy, "dy", (rows, cols), dt, dev)
    _need(y, "y", (rows, cols), dt, dev)
    dx = torch.empty_like(dy) if dx is None else _need(dx, "dx", (rows, cols), dt, dev)
    name = f"ln_softmax_bwd_{sfx}"
    _check(name, getattr(lib(), name)(_ptr(dy), _ptr(y), float(scale), rows, cols, _ptr(dx),
                                      _stream(stream)))
    return dx


def xent(logits, targets, alpha: float = 0.0, dloss: float = 1.0, losses=None, dlogits=None,
         want_losses: bool = True, want_grad: bool = True, in_place: bool = False, stream=None):
    """Fused cross-entropy with label smoothing.  logits: [rows, V]; targets: int32 [rows].
    Returns (losses, dlogits): losses fp32 [rows] = -sum p log softmax(logits), dlogits =
    dloss * (softmax(logits) - p), p = (1 - alpha) onehot + alpha / V.  ``in_place`` writes
    the gradient over the logits."""
    import torch
    if logits.dim() != 2:
        raise ValueError("logits must be 2-D [rows, V]")
    rows, V = logits.shape
    dt, dev = logits.dtype, logits.device
    sfx = _suffix(dt)
    _need(logits, "logits", (rows, V), dt, dev)
    _need(targets, "targets", (rows,), torch.int32, dev)
    if want_losses and losses is None:
        losses = torch.empty(rows, dtype=torch.float32, device=dev)
    elif losses is not None:
        _need(losses, "losses", (rows,), torch.float32, dev)
    if in_place:
        dlogits = logits
    elif want_grad and dlogits is None:
        dlogits = torch.empty_like(logits)
    elif dlogits is not None:
        _need(dlogits, "dlogits", (rows, V), dt, dev)
    name = f"ln_xent_{sfx}"
    _check(name, getattr(lib(), name)(_ptr(logits), _ptr(targets), rows, V, float(alpha),
                                      float(dloss), _ptr(losses), _ptr(dlogits), _stream(stream)))
    return losses, dlogits


def dropout_keep_bytes(rows: int, cols: int) -> int:
    """Bytes of the stored keep bits of a [rows, cols] prologue: rows * ceil(cols / 8)."""
    return int(lib().ln_dropout_keep_bytes(rows, cols))


def fwd_bias_dropout(h, bias, res, gamma, beta, eps: float = 1e-5, p: float = 0.1, seed: int = 0,
                     offset: int = 0, out=None, res_out=None, mean=None, rstd=None, keep=None,
                     stream=None):
    """LayerNorm forward with the bias + dropout + residual prologue: s = res + keep * (h +
    bias) / (1 - p) (stored as res_out), then LN(s).  The dropout mask is a function of
    (seed, offset, element index); given ``keep`` (a uint8 tensor of
    :func:`dropout_keep_bytes` bytes), the decisions are also stored there as bits, for
    :func:`dropout_bwd`.  Returns (out, res_out, mean, rstd)."""
    import torch
    if h.dim() != 2:
        raise ValueError("h must be 2-D [rows, cols]")
    rows, cols = h.shape
    dt, dev = h.dtype, h.device
    sfx = _suffix(dt)
    _need(h, "h", (rows, cols), dt, dev)
    _need(res, "res", (rows, cols), dt, dev)
    for name, t in (("bias", bias), ("gamma", gamma), ("beta", beta)):
        _need(t, name, (cols,), dt, dev)
    out = torch.empty_like(h) if out is None else _need(out, "out", (rows, cols), dt, dev)
    res_out = torch.empty_like(h) if res_out is None else _need(res_out, "res_out", (rows, cols), dt, dev)
    mean = (torch.empty(rows, dtype=torch.float32, device=dev) if mean is None
            else _need(mean, "mean", (rows,), torch.float32, dev))
    rstd = (torch.empty(rows, dtype=torch.float32, device=dev) if rstd is None
            else _need(rstd, "rstd", (rows,), torch.float32, dev))
    args = [_ptr(h), _ptr(bias), _ptr(res), _ptr(gamma), _ptr(beta), float(eps), float(p),
            int(seed), int(offset), rows, cols, _ptr(out), _ptr(res_out), _ptr(mean), _ptr(rstd)]
    if keep is None:
        name = f"ln_fwd_bias_dropout_{sfx}"
    else:
        name = f"ln_fwd_bias_dropout_keep_{sfx}"
        args.append(_ptr(_keep_bytes(keep, rows, cols, dev)))
    _check(name, getattr(lib(), name)(*args, _stream(stream)))
    return out, res_out, mean, rstd


def _keep_bytes(keep, rows, cols, dev):
    import torch
    return _need(keep, "keep", (dropout_keep_bytes(rows, cols),), torch.uint8, dev)


def dropout_bwd(ds, p: float, seed: int = 0, offset: int = 0, dh=None, dbias=None,
                workspace=None, keep=None, stream=None):
    """Backward of the prologue: dh = ds * keep / (1 - p), dbias = sum over rows of dh (ds:
    the gradient with respect to s, i.e. :func:`bwd`'s dx); keep regenerated from (seed,
    offset), or read from the bits a :func:`fwd_bias_dropout` call with ``keep`` stored.
    Returns (dh, dbias)."""
    import torch
    if ds.dim() != 2:
        raise ValueError("ds must be 2-D [rows, cols]")
    rows, cols = ds.shape
    dt, dev = ds.dtype, ds.device
    sfx = _suffix(dt)
    _need(ds, "ds", (rows, cols), dt, dev)
    dh = torch.empty_like(ds) if dh is None else _need(dh, "dh", (rows, cols), dt, dev)
    dbias = (torch.empty(cols, dtype=dt, device=dev) if dbias is None
             else _need(dbias, "dbias", (cols,), dt, dev))
    if keep is None:
        kind, src = "", [int(seed), int(offset)]
    else:
        kind, src = "keep_", [_ptr(_keep_bytes(keep, rows, cols, dev))]
    args = [_ptr(ds), float(p), *src, rows, cols, _ptr(dh), _ptr(dbias)]
    if workspace is None:
        name = f"ln_dropout_bwd_{kind}{sfx}"
        _check(name, getattr(lib(), name)(*args, _stream(stream)))
    else:
        nbytes = workspace.numel() * workspace.element_size()
        name = f"ln_dropout_bwd_{kind}{sfx}_ws"
        _check(name, getattr(lib(), name)(*args, _ptr(workspace), nbytes, _stream(stream)))
    return dh, dbias
