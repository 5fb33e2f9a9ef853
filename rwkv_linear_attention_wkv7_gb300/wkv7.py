"""Thin Python binding of libwkv7 (the C ABI in include/wkv7.h).

Argument marshalling only: torch supplies device memory and the current CUDA
stream, every step of the recurrence runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing or the device is not an
sm_103a GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import torch

from . import _build

HEAD_SIZE = 64
WKV7_F32, WKV7_BF16 = 0, 1
_CODES = {0: "WKV7_OK", -1: "WKV7_EINVAL", -2: "WKV7_ECUDA", -3: "WKV7_EUNSUPPORTED"}
_lib = None


class WKV7Error(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} -> {_CODES.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libwkv7.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"libwkv7.so not built at {path}; run rwkv_linear_attention_wkv7_gb300.build()")
        _lib = load(path)
    return _lib


def load(path: str) -> ctypes.CDLL:
    """Open a build of the library at ``path`` with the C ABI's signatures declared."""
    L = ctypes.CDLL(path)
    vp, ci, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    L.wkv7_ckpt_count.argtypes = [ci, ci]
    L.wkv7_ckpt_count.restype = ci
    L.wkv7_factor_floats.argtypes = [ci]
    L.wkv7_factor_floats.restype = ctypes.c_longlong
    L.wkv7_forward.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [fp, fp, fp, fp, fp, ci, vp]
    L.wkv7_forward.restype = ci
    L.wkv7_backward.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [fp, fp, ci, fp, fp] + [fp] * 7 + [vp]
    L.wkv7_backward.restype = ci
    L.wkv7_timesplit_workspace_floats.argtypes = [ci, ci, ci, ci]
    L.wkv7_timesplit_workspace_floats.restype = ctypes.c_longlong
    L.wkv7_segment_scan.argtypes = [ci, ci, ci, fp, fp, fp, fp, fp, ci, vp]
    L.wkv7_segment_scan.restype = ci
    L.wkv7_forward_timesplit.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [fp, fp, fp, ci, fp, vp]
    L.wkv7_forward_timesplit.restype = ci
    L.wkv7_backward_timesplit.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [fp, fp] + [fp] * 7 + [ci, fp, vp]
    L.wkv7_backward_timesplit.restype = ci
    L.wkv7_forward_backward_blocks.argtypes = [ci, ci, ci, ci]
    L.wkv7_forward_backward_blocks.restype = ci
    L.wkv7_forward_state.argtypes = [ci, ci, ci, ci, ci] + [vp] * 5 + [fp, fp, vp]
    L.wkv7_forward_state.restype = ci
    L.wkv7_backward_state.argtypes = [ci, ci, ci, ci, ci] + [vp] * 4 + [fp] * 4 + [vp]
    L.wkv7_backward_state.restype = ci
    L.wkv7_forward_fused.argtypes = L.wkv7_forward.argtypes
    L.wkv7_forward_fused.restype = ci
    L.wkv7_backward_fused.argtypes = L.wkv7_backward.argtypes
    L.wkv7_backward_fused.restype = ci
    L.wkv7_gn_workspace_floats.argtypes = [ci, ci]
    L.wkv7_gn_workspace_floats.restype = ctypes.c_longlong
    L.wkv7_forward_gn.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [fp] * 4 + [fp] * 5 + [ci, vp]
    L.wkv7_forward_gn.restype = ci
    L.wkv7_backward_gn.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [fp, fp, ci] + [fp] * 5 + [fp] * 7 + [fp] * 4 + [vp]
    L.wkv7_backward_gn.restype = ci
    L.wkv7_forward_backward.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [fp] * 3 + [fp] * 4 + [fp] * 7 + [ci, vp]
    L.wkv7_forward_backward.restype = ci
    L.wkv7_forward_backward_fused.argtypes = L.wkv7_forward_backward.argtypes
    L.wkv7_forward_backward_fused.restype = ci
    L.wkv7_forward_backward_gn.argtypes = ([ci, ci, ci, ci, ci] + [vp] * 6 + [fp] * 3 + [fp] * 3 + [fp] * 5 + [fp] * 7 +
                                           [fp] * 3 + [fp, ci, vp])
    L.wkv7_forward_backward_gn.restype = ci
    L.wkv7_decode_step.argtypes = [ci, ci, ci, ci] + [vp] * 6 + [fp, fp, vp]
    L.wkv7_decode_step.restype = ci
    L.wkv7_async_status.argtypes = []
    L.wkv7_async_status.restype = ci
    L.wkv7_last_error.argtypes = []
    L.wkv7_last_error.restype = ctypes.c_char_p
    return L


def last_error() -> str:
    return lib().wkv7_last_error().decode()


def _check(fn: str, rc: int):
    if rc != 0:
        raise WKV7Error(fn, rc, last_error())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return WKV7_F32
    if t.dtype == torch.bfloat16:
        return WKV7_BF16
    raise TypeError(f"r, w, k, v, a, b must be float32 or bfloat16 (got {t.dtype})")


def _check_inputs(xs):
    r = xs[0]
    if r.dim() != 4 or r.shape[-1] != HEAD_SIZE:
        raise ValueError(f"inputs must be [B][T][H][{HEAD_SIZE}] (got {tuple(r.shape)})")
    for x in xs:
        if x.shape != r.shape or x.dtype != r.dtype or x.device != r.device:
            raise ValueError("r, w, k, v, a, b must share shape, dtype and device")
        if not x.is_contiguous():
            raise ValueError("inputs must be contiguous")
    if r.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")


def _f32(t, shape, device, name):
    if t is None:
        return None
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape) or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 {tuple(shape)} tensor on {device}")
    return t


def async_status() -> None:
    """Raise if a kernel's bounded wait on its bulk copies ran out since the
    last check (waits for the device to finish its work)."""
    _check("wkv7_async_status", lib().wkv7_async_status())


def ckpt_count(T: int, L: int) -> int:
    return lib().wkv7_ckpt_count(T, L)


def factor_floats(T: int) -> int:
    """Floats per (b, h) of the forward's per-chunk factor cache."""
    return lib().wkv7_factor_floats(T)


def forward(r, w, k, v, a, b, s0=None, L: int = 16, want_ckpt: bool = True, want_sT: bool = True,
            want_factors: bool = False, out: Optional[Dict[str, torch.Tensor]] = None, stream=None,
            _entry: str = "wkv7_forward"):
    """Run the recurrence over [B][T][H][64] inputs.

    Returns (y, sT, ckpt), or (y, sT, ckpt, factors) with ``want_factors``
    (the per-chunk factor cache for ``backward``; needs L == 16); sT / ckpt
    are None when not requested.  ``out`` may hold preallocated 'y', 'sT',
    'ckpt', 'factors' tensors.
    """
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    sshape = (B, H, N, N)
    out = out or {}
    y = out.get("y") if out.get("y") is not None else torch.empty((B, T, H, N), device=dev, dtype=torch.float32)
    sT = (out.get("sT") if out.get("sT") is not None else torch.empty(sshape, device=dev)) if want_sT else None
    nck = ckpt_count(T, L) if L >= 1 else -1
    ck = None
    if want_ckpt and nck >= 0:
        ck = out.get("ckpt") if out.get("ckpt") is not None else torch.empty((B, H, nck, N, N), device=dev)
    fac = None
    if want_factors:
        nf = factor_floats(T)
        fac = out.get("factors") if out.get("factors") is not None else torch.empty((B, H, max(nf, 0)), device=dev)
        _f32(fac, (B, H, nf), dev, "factors")
    _f32(y, (B, T, H, N), dev, "y")
    _f32(s0, sshape, dev, "s0")
    rc = getattr(lib(), _entry)(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(s0), _ptr(y), _ptr(sT), _ptr(ck),
                                _ptr(fac), L, _stream(stream))
    _check(_entry, rc)
    return (y, sT, ck, fac) if want_factors else (y, sT, ck)


GRAD_NAMES = ("dr", "dw", "dk", "dv", "da", "db")


def backward(r, w, k, v, a, b, ckpt, dy, dsT=None, L: int = 16, want_ds0: bool = True, factors=None,
             out: Optional[Dict[str, torch.Tensor]] = None, stream=None, _entry: str = "wkv7_backward",
             _names=None) -> Dict[str, torch.Tensor]:
    """Gradients of sum(y*dy) + sum(sT*dsT) w.r.t. r, w, k, v, a, b and s0.

    ``factors`` is the cache of the forward call that wrote ``ckpt`` (or None
    to recompute those per-chunk quantities)."""
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    out = out or {}
    names = _names or GRAD_NAMES
    g = {n: out.get(n) if out.get(n) is not None else torch.empty((B, T, H, N), device=dev) for n in names}
    g["ds0"] = (out.get("ds0") if out.get("ds0") is not None else torch.empty((B, H, N, N), device=dev)) if want_ds0 else None
    _f32(dy, (B, T, H, N), dev, "dy")
    _f32(dsT, (B, H, N, N), dev, "dsT")
    if factors is not None:
        _f32(factors, (B, H, factor_floats(T)), dev, "factors")
    rc = getattr(lib(), _entry)(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(ckpt), _ptr(factors), L,
                                _ptr(dy), _ptr(dsT),
                                *(_ptr(g[n]) for n in names), _ptr(g["ds0"]), _stream(stream))
    _check(_entry, rc)
    return g


def forward_backward_blocks(B: int, T: int, H: int, nsplit: int = 0) -> int:
    """Blocks of batch rows a one-call step with these sizes and ``nsplit`` runs
    (each launches one forward and one backward)."""
    n = lib().wkv7_forward_backward_blocks(B, T, H, nsplit)
    if n < 1:
        raise ValueError(f"bad sizes or nsplit (B={B}, T={T}, H={H}, nsplit={nsplit})")
    return n


def forward_backward(r, w, k, v, a, b, dy, s0=None, dsT=None, want_factors: bool = True, nsplit: int = 0,
                     out: Optional[Dict[str, torch.Tensor]] = None, stream=None, _entry: str = "wkv7_forward_backward",
                     _names=None) -> Dict[str, torch.Tensor]:
    """One training step through wkv7_forward_backward: the forward (checkpoint
    stride 16, and the factor cache with ``want_factors``) and the backward,
    as ``nsplit`` concurrent blocks of batch rows (0: the library's default).
    Returns a dict with 'y', 'sT', 'ckpt', 'factors' (or None) and the
    gradients 'dr' .. 'db', 'ds0'; ``out`` may hold any of them preallocated."""
    names = _names or GRAD_NAMES
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    out = out or {}
    sshape = (B, H, N, N)

    def get(name, shape):
        t = out.get(name)
        return t if t is not None else torch.empty(shape, device=dev)

    res = {"y": get("y", (B, T, H, N)), "sT": get("sT", sshape), "ckpt": get("ckpt", (B, H, ckpt_count(T, 16), N, N)),
           "factors": get("factors", (B, H, factor_floats(T))) if want_factors else None}
    for n in names:
        res[n] = get(n, (B, T, H, N))
    res["ds0"] = get("ds0", sshape)
    for n in ("y",) + names:
        _f32(res[n], (B, T, H, N), dev, n)
    _f32(res["ckpt"], (B, H, ckpt_count(T, 16), N, N), dev, "ckpt")
    if want_factors:
        _f32(res["factors"], (B, H, factor_floats(T)), dev, "factors")
    for n, t in (("sT", res["sT"]), ("ds0", res["ds0"]), ("s0", s0), ("dsT", dsT)):
        _f32(t, sshape, dev, n)
    _f32(dy, (B, T, H, N), dev, "dy")
    rc = getattr(lib(), _entry)(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(s0), _ptr(dy), _ptr(dsT),
                                _ptr(res["y"]), _ptr(res["sT"]), _ptr(res["ckpt"]), _ptr(res["factors"]),
                                *(_ptr(res[n]) for n in names), _ptr(res["ds0"]), int(nsplit), _stream(stream))
    _check(_entry, rc)
    return res


def forward_backward_fused(r, w_pre, k, v, kk, avec, dy, s0=None, dsT=None, nsplit: int = 0,
                           out: Optional[Dict[str, torch.Tensor]] = None, stream=None) -> Dict[str, torch.Tensor]:
    """forward_backward through wkv7_forward_backward_fused: the producers fused
    in (inputs w_pre, kk, avec; gradients 'dw_pre', 'dkk', 'davec')."""
    return forward_backward(r, w_pre, k, v, kk, avec, dy, s0=s0, dsT=dsT, want_factors=True, nsplit=nsplit, out=out,
                            stream=stream, _entry="wkv7_forward_backward_fused", _names=FUSED_GRAD_NAMES)


FUSED_GRAD_NAMES = ("dr", "dw_pre", "dk", "dv", "dkk", "davec")


def forward_fused(r, w_pre, k, v, kk, avec, s0=None, L: int = 16, want_ckpt: bool = True, want_sT: bool = True,
                  want_factors: bool = False, out: Optional[Dict[str, torch.Tensor]] = None, stream=None):
    """``forward`` with the producers of w, a, b fused in: w = exp(-0.606531 sigmoid(w_pre)),
    a = -kk, b = kk * avec (computed as the inputs are staged).  Needs L % 16 == 0."""
    return forward(r, w_pre, k, v, kk, avec, s0=s0, L=L, want_ckpt=want_ckpt, want_sT=want_sT,
                   want_factors=want_factors, out=out, stream=stream, _entry="wkv7_forward_fused")


def backward_fused(r, w_pre, k, v, kk, avec, ckpt, dy, dsT=None, L: int = 16, want_ds0: bool = True, factors=None,
                   out: Optional[Dict[str, torch.Tensor]] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Gradients dr, dw_pre, dk, dv, dkk, davec (and ds0) of the fused inputs; needs L == 16 and
    the factor cache of the matching ``forward_fused`` call."""
    return backward(r, w_pre, k, v, kk, avec, ckpt, dy, dsT=dsT, L=L, want_ds0=want_ds0, factors=factors,
                    out=out, stream=stream, _entry="wkv7_backward_fused", _names=FUSED_GRAD_NAMES)


def forward_gn(r, w, k, v, a, b, gn_w, gn_b, r_k, s0=None, L: int = 16, want_factors: bool = True,
               out: Optional[Dict[str, torch.Tensor]] = None, stream=None):
    """The recurrence with the GroupNorm + bonus output epilogue fused in
    (gn_w, gn_b, r_k [H][64] fp32).  Returns (o, y, sT, ckpt, factors): o the
    epilogue's output, y the recurrence's (read back by ``backward_gn``)."""
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    out = out or {}
    for n, t in (("gn_w", gn_w), ("gn_b", gn_b), ("r_k", r_k)):
        _f32(t, (H, N), dev, n)
    y = out.get("y") if out.get("y") is not None else torch.empty((B, T, H, N), device=dev)
    o = out.get("o") if out.get("o") is not None else torch.empty((B, T, H, N), device=dev)
    sT = out.get("sT") if out.get("sT") is not None else torch.empty((B, H, N, N), device=dev)
    ck = out.get("ckpt") if out.get("ckpt") is not None else torch.empty((B, H, ckpt_count(T, L), N, N), device=dev)
    fac = None
    if want_factors:
        fac = out.get("factors") if out.get("factors") is not None else torch.empty((B, H, factor_floats(T)),
                                                                                  device=dev)
    _f32(s0, (B, H, N, N), dev, "s0")
    rc = lib().wkv7_forward_gn(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(s0), _ptr(gn_w), _ptr(gn_b), _ptr(r_k),
                               _ptr(y), _ptr(o), _ptr(sT), _ptr(ck), _ptr(fac), L, _stream(stream))
    _check("wkv7_forward_gn", rc)
    return o, y, sT, ck, fac


def gn_workspace_floats(B: int, H: int) -> int:
    return lib().wkv7_gn_workspace_floats(B, H)


def backward_gn(r, w, k, v, a, b, ckpt, factors, y, do, gn_w, r_k, dsT=None, L: int = 16, workspace=None,
                out: Optional[Dict[str, torch.Tensor]] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Gradients of sum(o * do) + sum(sT * dsT) through the epilogue and the
    recurrence: dr, dw, dk, dv, da, db, ds0 and dgn_w, dgn_b, dr_k ([H][64])."""
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    out = out or {}
    g = {n: out.get(n) if out.get(n) is not None else torch.empty((B, T, H, N), device=dev) for n in GRAD_NAMES}
    g["ds0"] = out.get("ds0") if out.get("ds0") is not None else torch.empty((B, H, N, N), device=dev)
    for n in ("dgn_w", "dgn_b", "dr_k"):
        g[n] = out.get(n) if out.get(n) is not None else torch.empty((H, N), device=dev)
    ws = workspace if workspace is not None else torch.empty(gn_workspace_floats(B, H), device=dev)
    _f32(y, (B, T, H, N), dev, "y")
    _f32(do, (B, T, H, N), dev, "do")
    _f32(dsT, (B, H, N, N), dev, "dsT")
    rc = lib().wkv7_backward_gn(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(ckpt), _ptr(factors), L, _ptr(y),
                                _ptr(do), _ptr(dsT), _ptr(gn_w), _ptr(r_k), *(_ptr(g[n]) for n in GRAD_NAMES),
                                _ptr(g["ds0"]), _ptr(g["dgn_w"]), _ptr(g["dgn_b"]), _ptr(g["dr_k"]), _ptr(ws),
                                _stream(stream))
    _check("wkv7_backward_gn", rc)
    return g


def forward_backward_gn(r, w, k, v, a, b, do, gn_w, gn_b, r_k, s0=None, dsT=None, nsplit: int = 0, workspace=None,
                        out: Optional[Dict[str, torch.Tensor]] = None, stream=None) -> Dict[str, torch.Tensor]:
    """One training step with the output epilogue through wkv7_forward_backward_gn.
    Returns 'o', 'y', 'sT', 'ckpt', 'factors', the gradients 'dr' .. 'db', 'ds0'
    and 'dgn_w', 'dgn_b', 'dr_k'; ``out`` may hold any of them preallocated."""
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    out = out or {}

    def get(name, shape):
        t = out.get(name)
        return t if t is not None else torch.empty(shape, device=dev)

    res = {n: get(n, (B, T, H, N)) for n in ("o", "y") + GRAD_NAMES}
    res.update(sT=get("sT", (B, H, N, N)), ds0=get("ds0", (B, H, N, N)),
               ckpt=get("ckpt", (B, H, ckpt_count(T, 16), N, N)), factors=get("factors", (B, H, factor_floats(T))))
    for n in ("dgn_w", "dgn_b", "dr_k"):
        res[n] = get(n, (H, N))
    ws = workspace if workspace is not None else torch.empty(gn_workspace_floats(B, H), device=dev)
    for n, t in (("gn_w", gn_w), ("gn_b", gn_b), ("r_k", r_k), ("dgn_w", res["dgn_w"]), ("dgn_b", res["dgn_b"]),
                 ("dr_k", res["dr_k"])):
        _f32(t, (H, N), dev, n)
    for n in ("o", "y") + GRAD_NAMES:
        _f32(res[n], (B, T, H, N), dev, n)
    _f32(do, (B, T, H, N), dev, "do")
    for n, t in (("s0", s0), ("dsT", dsT), ("sT", res["sT"]), ("ds0", res["ds0"])):
        _f32(t, (B, H, N, N), dev, n)
    _f32(res["ckpt"], (B, H, ckpt_count(T, 16), N, N), dev, "ckpt")
    _f32(res["factors"], (B, H, factor_floats(T)), dev, "factors")
    rc = lib().wkv7_forward_backward_gn(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(s0), _ptr(do), _ptr(dsT),
                                        _ptr(gn_w), _ptr(gn_b), _ptr(r_k), _ptr(res["y"]), _ptr(res["o"]),
                                        _ptr(res["sT"]), _ptr(res["ckpt"]), _ptr(res["factors"]),
                                        *(_ptr(res[n]) for n in GRAD_NAMES), _ptr(res["ds0"]), _ptr(res["dgn_w"]),
                                        _ptr(res["dgn_b"]), _ptr(res["dr_k"]), _ptr(ws), int(nsplit), _stream(stream))
    _check("wkv7_forward_backward_gn", rc)
    return res


def timesplit_workspace_floats(B: int, T: int, H: int, nseg: int) -> int:
    return lib().wkv7_timesplit_workspace_floats(B, T, H, nseg)


def forward_timesplit(r, w, k, v, a, b, s0=None, nseg: int = 1, workspace=None,
                      out: Optional[Dict[str, torch.Tensor]] = None, stream=None):
    """Forward with every sequence cut into ``nseg`` segments run side by side
    (T a multiple of 16 * nseg).  Returns (y, sT, workspace); pass the workspace
    to ``backward_timesplit`` with the same inputs."""
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    out = out or {}
    nws = timesplit_workspace_floats(B, T, H, nseg)
    if nws < 0:
        raise ValueError(f"T={T} is not a multiple of 16 * nseg (nseg={nseg})")
    ws = workspace if workspace is not None else torch.empty(max(nws, 1), device=dev)
    y = out.get("y") if out.get("y") is not None else torch.empty((B, T, H, N), device=dev)
    sT = out.get("sT") if out.get("sT") is not None else torch.empty((B, H, N, N), device=dev)
    _f32(s0, (B, H, N, N), dev, "s0")
    rc = lib().wkv7_forward_timesplit(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(s0), _ptr(y), _ptr(sT), nseg,
                                      _ptr(ws), _stream(stream))
    _check("wkv7_forward_timesplit", rc)
    return y, sT, ws


def backward_timesplit(r, w, k, v, a, b, dy, dsT=None, nseg: int = 1, workspace=None,
                       out: Optional[Dict[str, torch.Tensor]] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Gradients (as ``backward``) from the workspace of the matching ``forward_timesplit``."""
    xs = (r, w, k, v, a, b)
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    out = out or {}
    g = {n: out.get(n) if out.get(n) is not None else torch.empty((B, T, H, N), device=dev) for n in GRAD_NAMES}
    g["ds0"] = out.get("ds0") if out.get("ds0") is not None else torch.empty((B, H, N, N), device=dev)
    _f32(dy, (B, T, H, N), dev, "dy")
    _f32(dsT, (B, H, N, N), dev, "dsT")
    rc = lib().wkv7_backward_timesplit(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(dy), _ptr(dsT),
                                       *(_ptr(g[n]) for n in GRAD_NAMES), _ptr(g["ds0"]), nseg, _ptr(workspace),
                                       _stream(stream))
    _check("wkv7_backward_timesplit", rc)
    return g


def forward_state(w, k, v, a, b, s0=None, sT=None, stream=None) -> torch.Tensor:
    """sT of ``forward`` alone (no y, checkpoints or factors).  ``v=None`` reads
    v as zero (k is then not read): from s0 = I that is the transition product
    of the inputs' span, see wkv7_forward_state."""
    xs = [w, k if v is not None else w, v if v is not None else w, a, b]
    _check_inputs(xs)
    B, T, H, N = w.shape
    dev = w.device
    sT = sT if sT is not None else torch.empty((B, H, N, N), device=dev)
    _f32(sT, (B, H, N, N), dev, "sT")
    _f32(s0, (B, H, N, N), dev, "s0")
    ptrs = [_ptr(w), _ptr(k) if v is not None else None, _ptr(v), _ptr(a), _ptr(b)]
    rc = lib().wkv7_forward_state(B, T, H, N, _dtype_code(w), *ptrs, _ptr(s0), _ptr(sT), _stream(stream))
    _check("wkv7_forward_state", rc)
    return sT


def backward_state(r, w, a, b, factors, dy, dsT=None, ds0=None, stream=None) -> torch.Tensor:
    """ds0 of ``backward`` alone, from the forward's factor cache (no
    checkpoints; k and v do not enter it), see wkv7_backward_state."""
    xs = [r, w, a, b]
    _check_inputs(xs)
    B, T, H, N = r.shape
    dev = r.device
    ds0 = ds0 if ds0 is not None else torch.empty((B, H, N, N), device=dev)
    _f32(ds0, (B, H, N, N), dev, "ds0")
    _f32(dy, (B, T, H, N), dev, "dy")
    _f32(dsT, (B, H, N, N), dev, "dsT")
    _f32(factors, (B, H, factor_floats(T)), dev, "factors")
    rc = lib().wkv7_backward_state(B, T, H, N, _dtype_code(r), *map(_ptr, xs), _ptr(factors), _ptr(dy), _ptr(dsT),
                                   _ptr(ds0), _stream(stream))
    _check("wkv7_backward_state", rc)
    return ds0


def segment_scan(M, C, init=None, backward: bool = False, out=None, fin=None, stream=None):
    """The segment scan alone: M, C [B][nseg][H][64][64] fp32; returns (out, fin) with out_k the
    state entering segment k (forward) or the gradient arriving at its end (backward) and fin the
    final state / the gradient at the start (see wkv7_segment_scan)."""
    B, nseg, H, N, _ = M.shape
    dev = M.device
    _f32(M, (B, nseg, H, N, N), dev, "M")
    _f32(C, (B, nseg, H, N, N), dev, "C")
    _f32(init, (B, H, N, N), dev, "init")
    out = out if out is not None else torch.empty_like(M)
    fin = fin if fin is not None else torch.empty((B, H, N, N), device=dev)
    rc = lib().wkv7_segment_scan(B, H, nseg, _ptr(M), _ptr(C), _ptr(init), _ptr(out), _ptr(fin), int(backward),
                                 _stream(stream))
    _check("wkv7_segment_scan", rc)
    return out, fin


def decode_step(r, w, k, v, a, b, state, y=None, stream=None):
    """One token for each of B*H heads; vectors [B][H][64], ``state`` updated in place."""
    if r.dim() != 3 or r.shape[-1] != HEAD_SIZE:
        raise ValueError(f"decode vectors must be [B][H][{HEAD_SIZE}] (got {tuple(r.shape)})")
    for x in (r, w, k, v, a, b):
        if x.shape != r.shape or x.dtype != r.dtype or not x.is_contiguous() or x.device != r.device:
            raise ValueError("decode vectors must share shape, dtype, device and be contiguous")
    B, H, N = r.shape
    _f32(state, (B, H, N, N), r.device, "state")
    y = y if y is not None else torch.empty((B, H, N), device=r.device)
    rc = lib().wkv7_decode_step(B, H, N, _dtype_code(r), *map(_ptr, (r, w, k, v, a, b)), _ptr(state), _ptr(y),
                                _stream(stream))
    _check("wkv7_decode_step", rc)
    return y


class WKV7Function(torch.autograd.Function):
    """autograd wrapper: y, sT = wkv7(r, w, k, v, a, b, s0) with checkpoint stride L."""

    @staticmethod
    def forward(ctx, r, w, k, v, a, b, s0, L):
        y, sT, ck, fac = forward(r, w, k, v, a, b, s0=s0, L=L, want_factors=True) if L == 16 else (
            *forward(r, w, k, v, a, b, s0=s0, L=L), None)
        ctx.save_for_backward(r, w, k, v, a, b, ck, fac)
        ctx.L = L
        ctx.has_s0 = s0 is not None
        return y, sT

    @staticmethod
    def backward(ctx, dy, dsT):
        r, w, k, v, a, b, ck, fac = ctx.saved_tensors
        g = backward(r, w, k, v, a, b, ck, dy.contiguous().float(),
                     None if dsT is None else dsT.contiguous().float(), L=ctx.L, want_ds0=ctx.has_s0, factors=fac)
        cast = (lambda t: t.to(r.dtype)) if r.dtype != torch.float32 else (lambda t: t)
        return (*(cast(g[n]) for n in GRAD_NAMES), g["ds0"], None)


def wkv7(r, w, k, v, a, b, s0=None, L: int = 16) -> Tuple[torch.Tensor, torch.Tensor]:
    """Differentiable WKV7: returns (y, sT)."""
    return WKV7Function.apply(r, w, k, v, a, b, s0, L)
