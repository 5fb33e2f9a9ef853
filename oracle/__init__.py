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

# ---- the output epilogue after the recurrence ("Foundry/cuda_kernels/timemix.cu"
# page: k_groupnorm, then k_bonus; their backward halves k_bonus_bwd and
# k_groupnorm_bwd).  Per token and head, over the head's N recurrence outputs y:
#     mean = sum_j y_j / N,  var = sum_j (y_j - mean)^2 / N,  rstd = 1 / sqrt(var + 64e-5)
#     g_j = (y_j - mean) rstd gn_w[h][j] + gn_b[h][j]                 (k_groupnorm: one group per head)
#     s = sum_j r_j k_j r_k[h][j],   o_j = g_j + s v_j                  (k_bonus)
# with the GroupNorm's per-channel weight and bias gn_w, gn_b and the bonus
# weight r_k, each per channel c = h N + j.  Backward from do = dL/do:
#     ds = sum_j do_j v_j;  dv += do s;  dr += ds k r_k;  dk += ds r r_k;  d r_k = sum ds r k   (k_bonus_bwd)
#     xh = (y - mean) rstd;  dn = do gn_w
#     dy = rstd (dn - mean_j(dn) - xh mean_j(dn xh));  d gn_w = sum do xh;  d gn_b = sum do    (k_groupnorm_bwd)
# with the parameter gradients summed over every batch row and token.
# Readings: r, k, v here are the recurrence's own inputs (the page's R, K, V
# buffers feed both); the bonus is added after the GroupNorm, as the page
# launches them; the page's output gate after the bonus belongs to the model
# around and is not part of this epilogue.
GN_EPS = 64e-5


def gn_bonus(y, r, k, v, gn_w, gn_b, r_k):
    """(o, mean, rstd) in float64.  y, r, k, v [B][T][H][N]; gn_w, gn_b, r_k [H][N];
    mean and rstd [B][T][H]."""
    y, r, k, v, gn_w, gn_b, r_k = map(_f64, (y, r, k, v, gn_w, gn_b, r_k))
    n = y.shape[-1]
    mean = y.sum(axis=-1, keepdims=True) / n
    var = ((y - mean) ** 2).sum(axis=-1, keepdims=True) / n
    rstd = 1.0 / np.sqrt(var + GN_EPS)
    g = (y - mean) * rstd * gn_w + gn_b
    s = (r * k * r_k).sum(axis=-1, keepdims=True)
    return g + s * v, mean[..., 0], rstd[..., 0]


def gn_bonus_backward(y, r, k, v, gn_w, r_k, do):
    """Gradients through the epilogue from do = dL/do: dy (what the recurrence
    receives), the bonus's own terms dr, dk, dv (added to the recurrence's),
    and the parameter gradients dgn_w, dgn_b, dr_k [H][N]."""
    y, r, k, v, gn_w, r_k, do = map(_f64, (y, r, k, v, gn_w, r_k, do))
    n = y.shape[-1]
    s = (r * k * r_k).sum(axis=-1, keepdims=True)
    ds = (do * v).sum(axis=-1, keepdims=True)
    out = {"dv": do * s, "dr": ds * k * r_k, "dk": ds * r * r_k, "dr_k": (ds * r * k).sum(axis=(0, 1))}
    mean = y.sum(axis=-1, keepdims=True) / n
    var = ((y - mean) ** 2).sum(axis=-1, keepdims=True) / n
    rstd = 1.0 / np.sqrt(var + GN_EPS)
    xh = (y - mean) * rstd
    dn = do * gn_w
    out["dy"] = rstd * (dn - dn.sum(axis=-1, keepdims=True) / n - xh * (dn * xh).sum(axis=-1, keepdims=True) / n)
    out["dgn_w"] = (do * xh).sum(axis=(0, 1))
    out["dgn_b"] = do.sum(axis=(0, 1))
    return out


def _forward_gn(orc, r, w, k, v, a, b, gn_w, gn_b, r_k, s0=None, L: int = 16, want_ckpt: bool = True):
    y, sT, ck = orc.forward(r, w, k, v, a, b, s0=s0, L=L, want_ckpt=want_ckpt)
    o, _, _ = gn_bonus(y, r, k, v, gn_w, gn_b, r_k)
    return o, y, sT, ck


def _backward_gn(orc, r, w, k, v, a, b, gn_w, r_k, do, s0=None, dsT=None):
    y, _, _ = orc.forward(r, w, k, v, a, b, s0=s0, L=16, want_ckpt=False)
    e = gn_bonus_backward(y, r, k, v, gn_w, r_k, do)
    g = orc.backward(r, w, k, v, a, b, e["dy"], s0=s0, dsT=dsT)
    for n in ("dr", "dk", "dv"):
        g[n] = g[n] + e[n]
    g.update({n: e[n] for n in ("dgn_w", "dgn_b", "dr_k")})
    return g


OracleLib.forward_gn = lambda self, *a, **kw: _forward_gn(self, *a, **kw)
OracleLib.backward_gn = lambda self, *a, **kw: _backward_gn(self, *a, **kw)
OracleLib.forward_gn.__doc__ = ("Recurrence, then GroupNorm + bonus: returns (o, y, sT, ckpt) from "
                                "(r, w, k, v, a, b, gn_w, gn_b, r_k).")
OracleLib.backward_gn.__doc__ = ("Gradients of sum(o * do) + sum(sT * dsT): dr, dw, dk, dv, da, db, ds0 "
                                 "and dgn_w, dgn_b, dr_k; arguments (r, w, k, v, a, b, gn_w, r_k, do).")

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


def forward_gn(*args, **kw):
    return lib().forward_gn(*args, **kw)


def backward_gn(*args, **kw):
    return lib().backward_gn(*args, **kw)


def per_head(fn, heads, threads=None):
    """Run ``fn(b, h)`` for every (b, h) in ``heads`` on a thread pool.

    The C calls release the GIL, so independent heads run on separate cores.
    Results come back in the order of ``heads``.
    """
    threads = threads or os.cpu_count() or 1
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda bh: fn(*bh), heads))
