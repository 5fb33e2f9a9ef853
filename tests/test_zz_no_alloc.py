"""wkv7_forward_backward_noalloc, the entry point for callers that cannot
allocate device memory (fixed memory pools, real-time loops, bindings without
a CUDA allocator): it keeps the forward's factor cache in a fixed array inside
the library instead of a caller-owned buffer.

Checked through the C ABI against the ordinary entry points (wkv7_forward
writing a caller-owned factor cache, wkv7_backward reading it) on two calls in
a row with different inputs and lengths, so that whatever the first call left
in the shared array cannot leak into the second.  This file is collected last.
"""
import ctypes

import pytest
import torch

from rwkv_linear_attention_wkv7_gb300 import synthetic, wkv7
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from rwkv_linear_attention_wkv7_gb300 import build
    build()
    assert torch.cuda.is_available()
    L = wkv7.lib()
    vp, ci = ctypes.c_void_p, ctypes.c_int
    L.wkv7_forward_backward_noalloc.argtypes = [ci, ci, ci, ci, ci] + [vp] * 6 + [vp] * 3 + [vp] * 3 + [vp] * 7 + [vp]
    L.wkv7_forward_backward_noalloc.restype = ci
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(L, d, dtype_code):
    B, T, H, N = d["r"].shape
    dev = d["r"].device
    y = torch.empty((B, T, H, N), device=dev)
    sT = torch.empty((B, H, N, N), device=dev)
    ck = torch.empty((B, H, wkv7.ckpt_count(T, 16), N, N), device=dev)
    g = {n: torch.empty((B, T, H, N), device=dev) for n in parity.GRADS}
    g["ds0"] = torch.empty((B, H, N, N), device=dev)
    rc = L.wkv7_forward_backward_noalloc(B, T, H, N, dtype_code, *(_ptr(d[n]) for n in parity.INPUTS),
                                         _ptr(d["s0"]), _ptr(d["dy"]), _ptr(d["dsT"]), _ptr(y), _ptr(sT), _ptr(ck),
                                         *(_ptr(g[n]) for n in parity.GRADS), _ptr(g["ds0"]), None)
    assert rc == 0, wkv7.last_error()
    torch.cuda.synchronize()
    return {"y": y, "sT": sT, "ckpt": ck, **g}


def test_noalloc_matches_the_allocating_entry_points(lib):
    """Both paths launch the same kernels with the same factor cache layout, so
    every output must be bit-identical; the last case fills the whole array
    (B*H*ceil(T/16) at the limit) after smaller calls left their data in it."""
    limit = 4096  # WKV7_NOALLOC_MAX_CHUNK_HEADS
    cases = [synthetic.WorkloadSpec("noalloc_a", 2, 200, 3, dtype="bf16", s0_std=0.1, with_dsT=True, seed=21),
             synthetic.WorkloadSpec("noalloc_b", 1, 77, 5, dtype="f32", s0_std=0.1, with_dsT=True, seed=22),
             synthetic.WorkloadSpec("noalloc_full", 1, 16 * limit // 4, 4, dtype="bf16", s0_std=0.1,
                                    with_dsT=True, seed=23)]
    assert cases[-1].B * cases[-1].H * ((cases[-1].T + 15) // 16) == limit
    for spec in cases:  # calls in a row; each reuses the array the previous one filled
        d, _ = parity.inputs_on_device(spec)
        got = _noalloc(lib, d, 1 if spec.dtype == "bf16" else 0)
        ref = parity.run_gpu(d, L=16, factors=True)
        for k in ("y", "sT", "ckpt") + parity.GRADS + ("ds0",):
            assert torch.equal(got[k], ref[k]), (spec.name, k)


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    p = ctypes.c_void_p(4096)
    args = [64, 4096, 32, 64, 1] + [p] * 6 + [None, p, None, p, None, p] + [p] * 6 + [None, None]
    assert lib.wkv7_forward_backward_noalloc(*args) == -1
    assert "exceeds the no-alloc factor scratch" in wkv7.last_error()
    # one chunk-head past the limit (B = H = 1, ceil(T/16) = 4097)
    args = [1, 16 * 4097, 1, 64, 1] + [p] * 6 + [None, p, None, p, None, p] + [p] * 6 + [None, None]
    assert lib.wkv7_forward_backward_noalloc(*args) == -1
    assert "4097 exceeds" in wkv7.last_error()
