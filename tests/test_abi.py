"""The C-ABI library: it builds, loads, exports every symbol include/wkv7.h
declares, and rejects bad arguments on the host before anything is launched
(no GPU needed: none of these calls reaches a kernel)."""
import ctypes
import os
import re

import pytest
import torch

from rwkv_linear_attention_wkv7_gb300 import build, wkv7

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")
EINVAL, EUNSUPPORTED = -1, -3


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(wkv7_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build()
    return wkv7.lib()


def test_header_is_plain_c_and_cpp():
    """include/wkv7.h compiles on its own as C99 and as C++17, warnings as errors."""
    import shutil
    import subprocess
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "wkv7.h")
    for cc, lang, std in (("gcc", "c", "-std=c99"), ("g++", "c++", "-std=c++17")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not available")
        r = subprocess.run([cc, "-fsyntax-only", "-x", lang, std, "-Wall", "-Wextra", "-Werror", hdr],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("wkv7_forward", "wkv7_backward", "wkv7_decode_step", "wkv7_ckpt_count", "wkv7_factor_floats",
                     "wkv7_async_status", "wkv7_last_error", "wkv7_forward_fused", "wkv7_backward_fused",
                     "wkv7_forward_gn", "wkv7_backward_gn", "wkv7_gn_workspace_floats",
                     "wkv7_forward_backward", "wkv7_forward_backward_fused", "wkv7_forward_backward_gn",
                     "wkv7_forward_state", "wkv7_backward_state"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_ckpt_count(lib):
    assert lib.wkv7_ckpt_count(0, 16) == 0
    assert lib.wkv7_ckpt_count(17, 16) == 2
    assert lib.wkv7_ckpt_count(4096, 16) == 256
    assert lib.wkv7_ckpt_count(-1, 16) == -1
    assert lib.wkv7_ckpt_count(5, 0) == -1


def test_factor_floats(lib):
    assert lib.wkv7_factor_floats(0) == 0
    assert lib.wkv7_factor_floats(1) == 2048
    assert lib.wkv7_factor_floats(17) == 2 * 2048
    assert lib.wkv7_factor_floats(4096) == 256 * 2048
    assert lib.wkv7_factor_floats(-1) == -1


def _fwd(lib, B=1, T=4, H=1, N=64, dt=0, ptr=None, y=None, L=16, s0=None, fac=None):
    p = ctypes.c_void_p(4096) if ptr is None else ptr
    y = p if y is None else y
    return lib.wkv7_forward(B, T, H, N, dt, p, p, p, p, p, p, s0, y, None, None, fac, L, None)


def test_forward_rejects_bad_arguments(lib):
    assert _fwd(lib, N=63) == EINVAL and "N must be 64" in wkv7.last_error()
    assert _fwd(lib, B=0) == EINVAL
    assert _fwd(lib, T=-1) == EINVAL
    assert _fwd(lib, dt=7) == EINVAL
    assert _fwd(lib, L=0) == EINVAL
    assert _fwd(lib, ptr=ctypes.c_void_p(4100)) == EINVAL and "aligned" in wkv7.last_error()
    assert lib.wkv7_forward(1, 4, 1, 64, 0, None, *([ctypes.c_void_p(4096)] * 5), None,
                            ctypes.c_void_p(4096), None, None, None, 16, None) == EINVAL
    assert "r is NULL" in wkv7.last_error()
    assert _fwd(lib, s0=ctypes.c_void_p(4104)) == EINVAL
    assert _fwd(lib, fac=ctypes.c_void_p(4096), L=32) == EINVAL and "L == 16" in wkv7.last_error()
    assert _fwd(lib, fac=ctypes.c_void_p(4104)) == EINVAL and "factors" in wkv7.last_error()


def test_backward_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(4096)
    args = [1, 4, 1, 64, 0] + [p] * 6 + [p, None, 16, p, None] + [p] * 6 + [None, None]
    bad = list(args)
    bad[11] = None  # ckpt missing
    assert lib.wkv7_backward(*bad) == EINVAL and "ckpt" in wkv7.last_error()
    bad = list(args)
    bad[13] = 0  # L
    assert lib.wkv7_backward(*bad) == EINVAL
    bad = list(args)
    bad[18] = ctypes.c_void_p(4098)  # dk misaligned
    assert lib.wkv7_backward(*bad) == EINVAL
    bad = list(args)
    bad[12], bad[13] = p, 8  # factors with a stride other than 16
    assert lib.wkv7_backward(*bad) == EINVAL and "L == 16" in wkv7.last_error()


def test_fused_entry_points_reject_bad_arguments(lib):
    """The fused producers run on the chunked path only: the forward needs L a
    multiple of 16, the backward L == 16 and the forward's factor cache."""
    p = ctypes.c_void_p(4096)
    assert lib.wkv7_forward_fused(1, 4, 1, 64, 0, *([p] * 6), None, p, None, None, None, 8, None) == EUNSUPPORTED
    assert "multiple of 16" in wkv7.last_error()
    assert lib.wkv7_forward_fused(1, 4, 1, 64, 0, p, None, *([p] * 4), None, p, None, None, None, 16, None) == EINVAL
    assert "w_pre is NULL" in wkv7.last_error()
    args = [1, 4, 1, 64, 0] + [p] * 6 + [p, p, 16, p, None] + [p] * 6 + [None, None]
    bad = list(args)
    bad[12] = None  # no factor cache
    assert lib.wkv7_backward_fused(*bad) == EINVAL and "factor cache" in wkv7.last_error()
    bad = list(args)
    bad[21] = None  # davec missing
    assert lib.wkv7_backward_fused(*bad) == EINVAL and "davec is NULL" in wkv7.last_error()


def test_gn_entry_points_reject_bad_arguments(lib):
    """The fused output epilogue: forward needs its three weights, o and L a
    multiple of 16; backward needs L == 16, the factor cache, y, the weights,
    the parameter-gradient outputs and the workspace."""
    p = ctypes.c_void_p(4096)
    assert lib.wkv7_gn_workspace_floats(2, 3) == 2 * 3 * 3 * 64
    assert lib.wkv7_gn_workspace_floats(0, 3) == -1
    fwd = [1, 4, 1, 64, 0] + [p] * 6 + [None, p, p, p] + [p, p, None, None, None, 16, None]
    bad = list(fwd)
    bad[14] = None  # r_k
    assert lib.wkv7_forward_gn(*bad) == EINVAL and "required" in wkv7.last_error()
    bad = list(fwd)
    bad[20] = 8  # stride
    assert lib.wkv7_forward_gn(*bad) == EUNSUPPORTED and "multiple of 16" in wkv7.last_error()
    bad = list(fwd)
    bad[12] = ctypes.c_void_p(4100)  # gn_w misaligned
    assert lib.wkv7_forward_gn(*bad) == EINVAL and "gn_w" in wkv7.last_error()
    bwd = [1, 4, 1, 64, 0] + [p] * 6 + [p, p, 16, p, p, None, p, p] + [p] * 6 + [None] + [p] * 3 + [p, None]
    bad = list(bwd)
    bad[12] = None  # no factor cache
    assert lib.wkv7_backward_gn(*bad) == EINVAL and "factor cache" in wkv7.last_error()
    bad = list(bwd)
    bad[14] = None  # y
    assert lib.wkv7_backward_gn(*bad) == EINVAL and "y is NULL" in wkv7.last_error()
    bad = list(bwd)
    bad[29] = None  # workspace
    assert lib.wkv7_backward_gn(*bad) == EINVAL and "workspace" in wkv7.last_error()
    bad = list(bwd)
    bad[17] = None  # gn_w
    assert lib.wkv7_backward_gn(*bad) == EINVAL and "gn_w" in wkv7.last_error()


def test_forward_backward_rejects_bad_arguments(lib):
    """The one-call training step: nsplit in 0..4, dy and ckpt required,
    factors optional but aligned, N = 64; all before any device query."""
    p = ctypes.c_void_p(4096)
    args = [1, 4, 1, 64, 0] + [p] * 6 + [None, p, None] + [p, None, p, None] + [p] * 6 + [None, 0, None]
    for ns in (5, -1):
        bad = list(args)
        bad[25] = ns
        assert lib.wkv7_forward_backward(*bad) == EINVAL and "nsplit" in wkv7.last_error()
    bad = list(args)
    bad[12] = None  # dy
    assert lib.wkv7_forward_backward(*bad) == EINVAL and "dy" in wkv7.last_error()
    bad = list(args)
    bad[16] = None  # ckpt
    assert lib.wkv7_forward_backward(*bad) == EINVAL and "ckpt" in wkv7.last_error()
    bad = list(args)
    bad[17] = ctypes.c_void_p(4100)  # factors misaligned
    assert lib.wkv7_forward_backward(*bad) == EINVAL and "factors" in wkv7.last_error()
    bad = list(args)
    bad[3] = 32  # N
    assert lib.wkv7_forward_backward(*bad) == EINVAL
    # the fused form needs the factor cache, and names the fused arguments
    assert lib.wkv7_forward_backward_fused(*args) == EINVAL and "factor cache" in wkv7.last_error()
    good = list(args)
    good[17] = p
    bad = list(good)
    bad[6] = None  # w_pre
    assert lib.wkv7_forward_backward_fused(*bad) == EINVAL and "w_pre" in wkv7.last_error()
    # the epilogue form: its weights, parameter gradients and workspace are required
    gn = [1, 4, 1, 64, 0] + [p] * 6 + [None, p, None] + [p, p, p] + [p, p, None, p, p] + [p] * 6 + [None] + \
         [p, p, p] + [p, 0, None]
    for i, name in ((15, "gn_b"), (32, "workspace"), (29, "dgn_w")):
        bad = list(gn)
        bad[i] = None
        assert lib.wkv7_forward_backward_gn(*bad) == EINVAL and name in wkv7.last_error()
    bad = list(gn)
    bad[33] = 7
    assert lib.wkv7_forward_backward_gn(*bad) == EINVAL and "nsplit" in wkv7.last_error()


def test_state_passes_reject_bad_arguments(lib):
    """wkv7_forward_state needs sT (and k when v is given); wkv7_backward_state
    needs ds0 and the forward's factor cache."""
    p, odd = ctypes.c_void_p(4096), ctypes.c_void_p(4104)
    fwd = [1, 4, 1, 64, 0] + [p] * 5 + [None, p, None]
    bad = list(fwd)
    bad[11] = None
    assert lib.wkv7_forward_state(*bad) == EINVAL and "sT" in wkv7.last_error()
    bad = list(fwd)
    bad[6] = None  # k missing while v is given
    assert lib.wkv7_forward_state(*bad) == EINVAL and "k is NULL" in wkv7.last_error()
    bad = list(fwd)
    bad[10] = odd
    assert lib.wkv7_forward_state(*bad) == EINVAL and "aligned" in wkv7.last_error()
    bwd = [1, 4, 1, 64, 0] + [p] * 4 + [p, p, None, p, None]
    bad = list(bwd)
    bad[9] = None
    assert lib.wkv7_backward_state(*bad) == EINVAL and "factors" in wkv7.last_error()
    bad = list(bwd)
    bad[12] = None
    assert lib.wkv7_backward_state(*bad) == EINVAL and "ds0" in wkv7.last_error()
    bad = list(bwd)
    bad[3] = 32
    assert lib.wkv7_backward_state(*bad) == EINVAL and "N must be 64" in wkv7.last_error()


def test_forward_backward_blocks(lib):
    """The one-call step's block count: four blocks from 512 heads, two below,
    never more than the batch rows, one without tokens; -1 for bad arguments."""
    assert lib.wkv7_forward_backward_blocks(16, 4096, 32, 0) == 4
    assert lib.wkv7_forward_backward_blocks(8, 4096, 32, 0) == 2
    assert lib.wkv7_forward_backward_blocks(1, 4096, 32, 0) == 1
    assert lib.wkv7_forward_backward_blocks(3, 64, 2, 4) == 3
    assert lib.wkv7_forward_backward_blocks(16, 0, 32, 0) == 1
    assert lib.wkv7_forward_backward_blocks(16, 64, 32, 1) == 1
    assert lib.wkv7_forward_backward_blocks(0, 64, 32, 0) == -1
    assert lib.wkv7_forward_backward_blocks(4, 64, 32, 5) == -1
    assert lib.wkv7_forward_backward_blocks(4, -1, 32, 0) == -1


def test_decode_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(4096)
    assert lib.wkv7_decode_step(1, 1, 32, 0, *([p] * 6), p, p, None) == EINVAL
    assert lib.wkv7_decode_step(1, 1, 64, 0, *([p] * 6), None, p, None) == EINVAL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_no_gpu_is_reported_not_faked(lib):
    """Without a usable sm_103a device the library refuses; it has no CPU path."""
    assert _fwd(lib) == EUNSUPPORTED
    assert lib.wkv7_async_status() == EUNSUPPORTED
    assert "device" in wkv7.last_error()
