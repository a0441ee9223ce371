"""The C-ABI library on the CPU: it builds, loads, exports every symbol include/ln.h
declares, and rejects invalid arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import layernorm_ln_fwd_gb300 as ln
from layernorm_ln_fwd_gb300 import build as lnbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ln.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(ln_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    lnbuild.build()
    return ln.lib()


def test_header_declares_the_forward_and_backward_calls():
    names = _declared_functions()
    for n in ("ln_fwd_f32", "ln_fwd_bf16", "ln_bwd_f32", "ln_bwd_bf16"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} missing from libln.so"
    out = subprocess.run(["nm", "-D", "--defined-only", ln.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ln_[a-z0-9_]+)\b", out))
    assert set(names) <= exported
    # The binding knows the signature of every declared function, and nothing else.
    assert set(ln.SIGNATURES) == set(names)


def test_library_is_built_for_sm_103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(lnbuild.ARCH)


def test_status_strings(lib):
    for code, name in ln.STATUS.items():
        assert lib.ln_status_str(code).decode().startswith(name)
    assert lib.ln_version() >= 10000


NULL = None


def test_invalid_arguments_are_rejected_on_the_host(lib):
    p = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    # Missing required pointers.
    assert lib.ln_fwd_f32(NULL, NULL, p, p, 1e-5, 4, 4, p, NULL, p, p, NULL) == 1
    assert lib.ln_fwd_bf16(p, NULL, NULL, p, 1e-5, 4, 4, p, NULL, p, p, NULL) == 1
    assert lib.ln_bwd_f32(p, p, p, p, p, p, p, NULL, 4, 4, NULL) == 1
    assert lib.ln_bwd_bf16(NULL, p, p, p, p, p, p, p, 4, 4, NULL) == 1
    # Bad sizes and eps.
    assert lib.ln_fwd_f32(p, NULL, p, p, 1e-5, -1, 4, p, NULL, p, p, NULL) == 1
    assert lib.ln_fwd_f32(p, NULL, p, p, 1e-5, 4, 0, p, NULL, p, p, NULL) == 1
    assert lib.ln_fwd_f32(p, NULL, p, p, -1.0, 4, 4, p, NULL, p, p, NULL) == 1
    assert lib.ln_fwd_f32(p, NULL, p, p, float("nan"), 4, 4, p, NULL, p, p, NULL) == 1
    assert lib.ln_fwd_f32(p, NULL, p, p, float("inf"), 4, 4, p, NULL, p, p, NULL) == 1
    assert lib.ln_fwd_f32(p, NULL, p, p, 1e-5, 4, ln.MAX_COLS + 1, p, NULL, p, p, NULL) == 3
    assert lib.ln_fwd_bf16(p, NULL, p, p, 1e-5, 1 << 31, 8, p, NULL, p, p, NULL) == 3
    # LN_MAX_ROWS = 2^31 - 2^16: one more row is refused (row indices must stay in int range).
    assert lib.ln_fwd_bf16(p, NULL, p, p, 1e-5, 2**31 - 2**16 + 1, 8, p, NULL, p, p, NULL) == 3
    assert lib.ln_bwd_bf16(p, p, p, p, p, p, p, p, 2**31 - 2**16 + 1, 8, NULL) == 3
    assert lib.ln_bwd_f32(p, p, p, p, p, p, p, p, 4, ln.MAX_COLS + 1, NULL) == 3
    # rows == 0 is a forward no-op, needs no device, and accepts NULL row arrays.
    assert lib.ln_fwd_f32(p, NULL, p, p, 1e-5, 0, 4, p, NULL, p, p, NULL) == 0
    assert lib.ln_fwd_f32(NULL, NULL, NULL, NULL, 1e-5, 0, 4, NULL, NULL, NULL, NULL, NULL) == 0
    # The backward with rows == 0 still needs dgamma and dbeta (it zeroes them).
    assert lib.ln_bwd_f32(NULL, NULL, NULL, NULL, NULL, NULL, NULL, p, 0, 4, NULL) == 1
    # Caller-owned workspace: NULL and misaligned workspaces.
    assert lib.ln_bwd_f32_ws(p, p, p, p, p, p, p, p, 4, 4, NULL, 0, NULL) == 1
    assert lib.ln_bwd_bf16_ws(p, p, p, p, p, p, p, p, 4, 4, ctypes.c_void_p(272), 1 << 20,
                              NULL) == 2
    # Invalid sizes give no workspace size.
    assert lib.ln_bwd_workspace_bytes(4, 0) == 0
    assert lib.ln_bwd_workspace_bytes(-1, 4) == 0
    assert lib.ln_last_launch_count() == 0
    # RMSNorm: beta and mean do not exist, gamma and rrms are required.
    assert lib.ln_rms_fwd_f32(p, NULL, NULL, 1e-5, 4, 4, p, NULL, p, NULL) == 1
    assert lib.ln_rms_fwd_bf16(p, NULL, p, 1e-5, 4, 4, p, NULL, NULL, NULL) == 1
    assert lib.ln_rms_fwd_f32(p, NULL, p, -1.0, 4, 4, p, NULL, p, NULL) == 1
    assert lib.ln_rms_fwd_bf16(p, NULL, p, 1e-5, 4, ln.MAX_COLS + 1, p, NULL, p, NULL) == 3
    assert lib.ln_rms_bwd_f32(p, p, p, NULL, p, p, 4, 4, NULL) == 1
    assert lib.ln_rms_bwd_bf16(p, p, p, p, p, NULL, 4, 4, NULL) == 1
    assert lib.ln_rms_bwd_bf16_ws(p, p, p, p, p, p, 4, 4, ctypes.c_void_p(272), 1 << 20,
                                  NULL) == 2
    assert lib.ln_rms_fwd_f32(NULL, NULL, NULL, 1e-5, 0, 4, NULL, NULL, NULL, NULL) == 0


def test_stored_keep_bits_calls_are_checked_on_the_host(lib):
    p = ctypes.c_void_p(256)
    assert lib.ln_dropout_keep_bytes(4, 9) == 8  # rows padded to whole bytes
    assert lib.ln_dropout_keep_bytes(3, 16) == 6
    assert lib.ln_dropout_keep_bytes(4, 0) == 0
    assert lib.ln_dropout_keep_bytes(-1, 8) == 0
    # A missing keep buffer, or a bad p, is refused before anything is launched.
    assert lib.ln_fwd_bias_dropout_keep_f32(p, p, p, p, p, 1e-5, 0.1, 1, 2, 4, 8, p, p, p, p,
                                            NULL, NULL) == 1
    assert lib.ln_fwd_bias_dropout_keep_bf16(p, p, p, p, p, 1e-5, 1.0, 1, 2, 4, 8, p, p, p, p,
                                             p, NULL) == 1
    assert lib.ln_dropout_bwd_keep_f32(p, 0.1, NULL, 4, 8, p, p, NULL) == 1
    assert lib.ln_dropout_bwd_keep_bf16_ws(p, 0.1, p, 4, 8, p, p, ctypes.c_void_p(272), 1 << 20,
                                           NULL) == 2
    assert lib.ln_last_launch_count() == 0


def test_force_path_hook_round_trips(lib):
    prev = lib.ln_debug_force_path(ln.PATH_SCALAR)
    assert lib.ln_debug_force_path(ln.PATH_AUTO) == ln.PATH_SCALAR
    lib.ln_debug_force_path(prev)
    assert lib.ln_debug_force_path(99) == prev  # out-of-range selects automatic
    assert lib.ln_debug_force_path(prev) == ln.PATH_AUTO


def test_binding_checks_without_a_gpu():
    import torch
    x = torch.zeros(4, 8)
    with pytest.raises(TypeError):
        ln.fwd(x.double(), None, torch.zeros(8).double(), torch.zeros(8).double())
    with pytest.raises(ValueError):
        ln.fwd(x, None, torch.zeros(7), torch.zeros(8))
    with pytest.raises(ValueError):
        ln.fwd(x.t(), None, torch.zeros(4), torch.zeros(4))
