"""WKV7 oracle -- test infrastructure only.

A plain double-precision CPU statement of the RWKV-7 WKV7 recurrence
(forward, exact adjoint, single-token decode), written in C
(``wkv7_oracle.c``) and called through ctypes.  Only the test suite, the
smoke check and the bench's CPU-baseline leg import this package; the CUDA
library never does, and the two share no code.

Arrays are numpy float64, C-contiguous, in the layouts of the CUDA library:
token vectors [B][T][H][N], states [B][H][N][N], checkpoints
[B][H][ceil(T/L)][N][N].  Float inputs (numpy, or torch bf16/fp32 tensors)
are widened to float64, which is exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "wkv7_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_wkv7.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]


def compile_c(src_path: str, out_path: str) -> str:
    """gcc one C file into a shared library (atomic replace)."""
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src_path])
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE double, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_c(SOURCE, _LIB)
    return _LIB


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: bf16/fp32 -> fp64 is exact
        import torch
        x = x.detach().to(device="cpu", dtype=torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(x):
    if x is None:
        return None
    assert x.dtype == np.float64 and x.flags.c_contiguous
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class OracleLib:
    """ctypes front of one compiled copy of the oracle."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        dp = ctypes.POINTER(ctypes.c_double)
        ci = ctypes.c_int
        lib.oracle_ckpt_count.argtypes = [ci, ci]
        lib.oracle_wkv7_forward.argtypes = [ci, ci, ci, ci, ci] + [dp] * 10
        lib.oracle_wkv7_backward.argtypes = [ci, ci, ci, ci] + [dp] * 16
        lib.oracle_wkv7_decode_step.argtypes = [ci, ci, ci] + [dp] * 8
        for f in (lib.oracle_ckpt_count, lib.oracle_wkv7_forward,
                  lib.oracle_wkv7_backward, lib.oracle_wkv7_decode_step):
            f.restype = ci
        self._lib = lib

    def ckpt_count(self, T: int, L: int) -> int:
        return self._lib.oracle_ckpt_count(T, L)

    def forward(self, r, w, k, v, a, b, s0=None, L: int = 16, want_ckpt: bool = True):
        """Return (y, sT, ckpt) in float64.  Inputs [B][T][H][N]."""
        r, w, k, v, a, b, s0 = map(_f64, (r, w, k, v, a, b, s0))
        B, T, H, N = r.shape
        y = np.zeros_like(r)
        sT = np.zeros((B, H, N, N))
        ckpt = np.zeros((B, H, self.ckpt_count(T, L), N, N)) if want_ckpt else None
        rc = self._lib.oracle_wkv7_forward(B, T, H, N, L, _p(r), _p(w), _p(k), _p(v), _p(a),
                                           _p(b), _p(s0), _p(y), _p(sT), _p(ckpt))
        if rc != 0:
            raise RuntimeError(f"oracle_wkv7_forward failed ({rc})")
        return y, sT, ckpt

    def backward(self, r, w, k, v, a, b, dy, s0=None, dsT=None):
        """Return a dict of float64 gradients dr, dw, dk, dv, da, db, ds0."""
        r, w, k, v, a, b, dy, s0, dsT = map(_f64, (r, w, k, v, a, b, dy, s0, dsT))
        B, T, H, N = r.shape
        g = {n: np.zeros_like(r) for n in ("dr", "dw", "dk", "dv", "da", "db")}
        g["ds0"] = np.zeros((B, H, N, N))
        rc = self._lib.oracle_wkv7_backward(
            B, T, H, N, _p(r), _p(w), _p(k), _p(v), _p(a), _p(b), _p(s0), _p(dy), _p(dsT),
            _p(g["dr"]), _p(g["dw"]), _p(g["dk"]), _p(g["dv"]), _p(g["da"]), _p(g["db"]),
            _p(g["ds0"]))
        if rc != 0:
            raise RuntimeError(f"oracle_wkv7_backward failed ({rc})")
        return g

    def decode_step(self, r, w, k, v, a, b, state):
        """One token for every (b,h).  Vectors [B][H][N]; returns (y, new_state)."""
        r, w, k, v, a, b = map(_f64, (r, w, k, v, a, b))
        st = _f64(state).copy()
        B, H, N = r.shape
        y = np.zeros_like(r)
        rc = self._lib.oracle_wkv7_decode_step(B, H, N, _p(r), _p(w), _p(k), _p(v), _p(a),
                                               _p(b), _p(st), _p(y))
        if rc != 0:
            raise RuntimeError(f"oracle_wkv7_decode_step failed ({rc})")
        return y, st


# ---- producers and backward epilogues fused into the recurrence's entry points
# ("Foundry/cuda_kernels/timemix.cu" page: k_decay, k_composites, and their
# backward halves k_wdecay_bwd, k_comp_keymod).  The fused calls take the
# pre-activation of the decay, the normalised key kk and the in-context
# learning-rate gate avec in place of (w, a, b):
#     sigma = 1 / (1 + exp(-w_pre)),  w = exp(-DECAY * sigma)      (k_decay)
#     a = -kk,  b = kk * avec                                          (k_composites)
# and return their gradients in place of (dw, da, db):
#     d w_pre = dw * w * (-DECAY) * sigma * (1 - sigma)               (k_wdecay_bwd)
#     d kk = -da + avec * db,  d avec = kk * db                        (k_comp_keymod, the
#         terms through a and b; its key-modulation terms belong to the model around)
# Reading: w_pre is the whole pre-activation (the page adds a per-channel bias
# w0 to the LoRA output before the sigmoid; the sum is the input here).
DECAY = 0.606531  # the decay scale of k_decay (e^{-1/2})


def producers(w_pre, kk, avec):
    """(w, a, b, sigma) in float64 from the fused inputs."""
    w_pre, kk, avec = map(_f64, (w_pre, kk, avec))
    with np.errstate(over="ignore"):
        sigma = 1.0 / (1.0 + np.exp(-w_pre))
    return np.exp(-DECAY * sigma), -kk, kk * avec, sigma


def epilogue(g, w, sigma, kk, avec):
    """Gradients of the fused inputs from those of (w, a, b)."""
    kk, avec = _f64(kk), _f64(avec)
    return {"dr": g["dr"], "dw_pre": g["dw"] * w * (-DECAY) * sigma * (1.0 - sigma), "dk": g["dk"],
            "dv": g["dv"], "dkk": -g["da"] + avec * g["db"], "davec": kk * g["db"], "ds0": g["ds0"]}


def _forward_fused(orc, r, w_pre, k, v, kk, avec, s0=None, L: int = 16, want_ckpt: bool = True):
    w, a, b, _ = producers(w_pre, kk, avec)
    return orc.forward(r, w, k, v, a, b, s0=s0, L=L, want_ckpt=want_ckpt)


def _backward_fused(orc, r, w_pre, k, v, kk, avec, dy, s0=None, dsT=None):
    w, a, b, sigma = producers(w_pre, kk, avec)
    return epilogue(orc.backward(r, w, k, v, a, b, dy, s0=s0, dsT=dsT), w, sigma, kk, avec)


OracleLib.forward_fused = lambda self, *a, **kw: _forward_fused(self, *a, **kw)
OracleLib.backward_fused = lambda self, *a, **kw: _backward_fused(self, *a, **kw)
OracleLib.forward_fused.__doc__ = "Forward from (r, w_pre, k, v, kk, avec); returns (y, sT, ckpt)."
OracleLib.backward_fused.__doc__ = ("Gradients dr, dw_pre, dk, dv, dkk, davec, ds0 of the fused inputs "
                                    "(same arguments as backward, with w_pre, kk, avec).")

_default = None


def lib() -> OracleLib:
    """The oracle compiled from ``wkv7_oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def ckpt_count(T, L):
    return lib().ckpt_count(T, L)


def forward(*args, **kw):
    return lib().forward(*args, **kw)


def backward(*args, **kw):
    return lib().backward(*args, **kw)


def decode_step(*args, **kw):
    return lib().decode_step(*args, **kw)


def forward_fused(*args, **kw):
    return lib().forward_fused(*args, **kw)


def backward_fused(*args, **kw):
    return lib().backward_fused(*args, **kw)


def per_head(fn, heads, threads=None):
    """Run ``fn(b, h)`` for every (b, h) in ``heads`` on a thread pool.

    The C calls release the GIL, so independent heads run on separate cores.
    Results come back in the order of ``heads``.
    """
    threads = threads or os.cpu_count() or 1
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda bh: fn(*bh), heads))
