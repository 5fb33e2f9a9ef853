"""The time-split entry points: every sequence cut into segments that run side
by side.  On the CPU the decomposition itself is checked with the oracle as
the segment solver (the recurrence is affine in a segment's start state); on
the GPU the library's time-split calls are checked against the oracle run
over the whole sequence."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from rwkv_linear_attention_wkv7_gb300 import build, synthetic, wkv7
from tests import parity

EINVAL = -1


def _segments(x, nseg):  # [B][T][H][N] -> [B*nseg][T/nseg][H][N]
    B, T, H, N = x.shape
    return x.reshape(B * nseg, T // nseg, H, N)


def _seg_states(s, B, nseg, H):  # [B*nseg][H][N][N] -> [B][nseg][H][N][N]
    return s.reshape(B, nseg, H, 64, 64)


def test_decomposition_with_the_oracle():
    """Forward: M_k from I with v = 0, Z_k from 0, S_{k+1} = S_k M_k + Z_k, then
    each segment from S_k reproduces the whole-sequence y and sT.  Backward:
    D_k with no gradient at the segment end, G_{k-1} = D_k + G_k M_k^T, then
    each segment with G_k reproduces every gradient and ds0."""
    spec = synthetic.WorkloadSpec("split", 2, 48, 2, s0_std=0.1, with_dsT=True, seed=8)
    x = {n: (None if t is None else t.double().numpy()) for n, t in synthetic.make_inputs(spec).items()}
    B, T, H, nseg = 2, 48, 2, 3
    names = parity.INPUTS
    seg = {n: _segments(x[n], nseg) for n in names + ("dy",)}
    eye = np.broadcast_to(np.eye(64), (B * nseg, H, 64, 64)).copy()
    _, M, _ = oracle.forward(*(seg[n] if n != "v" else np.zeros_like(seg["v"]) for n in names), s0=eye, L=16)
    _, Z, _ = oracle.forward(*(seg[n] for n in names), L=16)
    M, Z = _seg_states(M, B, nseg, H), _seg_states(Z, B, nseg, H)
    S = np.zeros((B, nseg, H, 64, 64))
    cur = x["s0"]
    for k in range(nseg):
        S[:, k] = cur
        cur = np.einsum("bhij,bhjk->bhik", cur, M[:, k]) + Z[:, k]
    y, _, _ = oracle.forward(*(seg[n] for n in names), s0=S.reshape(B * nseg, H, 64, 64), L=16)
    ref_y, ref_sT, _ = oracle.forward(*(x[n] for n in names), s0=x["s0"], L=16)
    assert parity.max_rel(y.reshape(x["r"].shape), ref_y) < 1e-12
    assert parity.max_rel(cur, ref_sT) < 1e-12

    s0s = S.reshape(B * nseg, H, 64, 64)
    D = oracle.backward(*(seg[n] for n in names), seg["dy"], s0=s0s)["ds0"]
    D = _seg_states(D, B, nseg, H)
    G = np.zeros((B, nseg, H, 64, 64))
    g = x["dsT"]
    for k in range(nseg - 1, -1, -1):
        G[:, k] = g
        g = D[:, k] + np.einsum("bhij,bhkj->bhik", g, M[:, k])
    got = oracle.backward(*(seg[n] for n in names), seg["dy"], s0=s0s, dsT=G.reshape(B * nseg, H, 64, 64))
    ref = oracle.backward(*(x[n] for n in names), x["dy"], s0=x["s0"], dsT=x["dsT"])
    for n in parity.GRADS:
        assert parity.max_rel(got[n].reshape(x["r"].shape), ref[n]) < 1e-11, n
    assert parity.max_rel(g, ref["ds0"]) < 1e-11


def test_workspace_size_and_argument_errors():
    build()
    lib = wkv7.lib()
    assert lib.wkv7_timesplit_workspace_floats(1, 100, 2, 4) == -1  # T not a multiple of 16 * nseg
    assert lib.wkv7_timesplit_workspace_floats(1, 128, 2, 0) == -1
    n = lib.wkv7_timesplit_workspace_floats(1, 128, 2, 4)
    assert n == 6 * 4 * 2 * 4096 + 4 * 2 * 2 * 4096 + 4 * 2 * 2 * 2048  # 6 state sets, checkpoints, factors
    p = ctypes.c_void_p(4096)
    fwd = lambda T, nseg, ws: lib.wkv7_forward_timesplit(1, T, 2, 64, 0, *([p] * 6), None, p, None, nseg, ws, None)
    assert fwd(100, 4, p) == EINVAL and "multiple of 16 * nseg" in wkv7.last_error()
    assert fwd(128, 0, p) == EINVAL
    assert fwd(128, 4, None) == EINVAL and "workspace" in wkv7.last_error()
    assert fwd(128, 4, ctypes.c_void_p(4100)) == EINVAL
    # the sizes, dtype and pointers are checked before anything is launched or zeroed
    bad_dtype = lib.wkv7_forward_timesplit(1, 128, 2, 64, 7, *([p] * 6), None, p, None, 4, p, None)
    assert bad_dtype == EINVAL and "dtype" in wkv7.last_error()
    no_y = lib.wkv7_forward_timesplit(1, 128, 2, 64, 0, *([p] * 6), None, None, None, 4, p, None)
    assert no_y == EINVAL and "y is NULL" in wkv7.last_error()
    odd_s0 = lib.wkv7_forward_timesplit(1, 128, 2, 64, 0, *([p] * 6), ctypes.c_void_p(4104), p, None, 4, p, None)
    assert odd_s0 == EINVAL and "s0" in wkv7.last_error()
    no_dr = lib.wkv7_backward_timesplit(1, 128, 2, 64, 0, *([p] * 6), p, None, None, *([p] * 5), None, 4, p, None)
    assert no_dr == EINVAL and "dr is NULL" in wkv7.last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,H,nseg,dtype", [(1, 512, 2, 4, "f32"), (2, 1024, 3, 8, "bf16"), (1, 256, 2, 1, "f32"),
                                              (1, 768, 2, 3, "bf16")])
def test_timesplit_matches_whole_sequence_oracle(B, T, H, nseg, dtype):
    build()
    spec = synthetic.WorkloadSpec("split", B, T, H, dtype=dtype, s0_std=0.1, with_dsT=True, seed=9)
    d, host = parity.inputs_on_device(spec)
    xs = [d[n] for n in parity.INPUTS]
    y, sT, ws = wkv7.forward_timesplit(*xs, s0=d["s0"], nseg=nseg)
    g = wkv7.backward_timesplit(*xs, d["dy"], dsT=d["dsT"], nseg=nseg, workspace=ws)
    torch.cuda.synchronize()
    wkv7.async_status()
    out = {"y": y, "sT": sT, **g}
    parity.check_heads(host, out, parity.all_heads(B, H), L=16)


def _scan_reference(M, C, init, backward):
    """The segment scan by its definition, in float64 on the CPU."""
    M, C = M.double().cpu(), C.double().cpu()
    B, nseg, H, N, _ = M.shape
    S = init.double().cpu().clone() if init is not None else torch.zeros((B, H, N, N), dtype=torch.float64)
    out = torch.empty_like(M)
    for step in range(nseg):
        k = nseg - 1 - step if backward else step
        out[:, k] = S
        S = C[:, k] + S @ (M[:, k].transpose(-1, -2) if backward else M[:, k])
    return out, S


@pytest.mark.gpu
@pytest.mark.parametrize("backward", [False, True])
@pytest.mark.parametrize("B,H,nseg,with_init", [(2, 3, 5, True), (1, 2, 1, False), (3, 1, 33, True)])
def test_segment_scan_against_its_definition(B, H, nseg, with_init, backward):
    """wkv7_segment_scan (split-operand tensor-core products, 16 rows per CTA)
    against S_{k+1} = C_k + S_k M_k (M_k^T backward) in float64.  The M_k are
    0.95 x random orthogonal matrices, so the states keep their scale over the
    steps; each split product is within about 3 * 2^-18 |a| |b| of the exact
    one, so 1e-4 of the largest entry bounds the error after 33 steps."""
    build()
    g = torch.Generator().manual_seed(5)
    Q, _ = torch.linalg.qr(torch.randn((B, nseg, H, 64, 64), generator=g, dtype=torch.float64))
    M = (0.95 * Q).float().contiguous()
    C = (0.1 * torch.randn((B, nseg, H, 64, 64), generator=g)).float()
    init = torch.randn((B, H, 64, 64), generator=g) if with_init else None
    out, fin = wkv7.segment_scan(M.cuda(), C.cuda(), init=None if init is None else init.cuda(), backward=backward)
    torch.cuda.synchronize()
    ref_out, ref_fin = _scan_reference(M, C, init, backward)
    for got, ref in ((out, ref_out), (fin, ref_fin)):
        err = (got.double().cpu() - ref).abs().max().item()
        assert err <= 1e-4 * ref.abs().max().item(), (err, ref.abs().max().item())
