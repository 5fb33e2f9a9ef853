"""Sequence parallelism across ranks (one process per GPU).

Every rank holds one contiguous span of the T axis of every sequence:
[B][T/world][H][64] inputs, rank order = time order.  The recurrence is
affine in the state a span starts from (S_end = S_start M + Z, M the product
of the span's transitions diag(w_t) + a_t b_t^T), so the only exchange is
two [B][H][64][64] matrices per rank and direction:

  forward   each rank: M (end state from I with v = 0) and Z (from 0) of its
            span; all-gather; the segment scan over the ranks gives every
            span's start state and the final state; each rank runs its span
            from its start state.
  backward  each rank: D, the gradient its span sends to its start when none
            arrives at its end; all-gather; the reverse scan gives the
            gradient arriving at every span's end and ds0; each rank runs its
            span's backward with that gradient.

Every step runs in the library's kernels (``CudaSpanSolver``); the matrices
cross ranks through ``torch.distributed.all_gather`` on the CPU (gloo) or
the GPU (nccl).  The solver is a parameter so that the exchange logic can be
exercised on the CPU with any stand-in of the same interface.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import torch
import torch.distributed as dist

from . import wkv7

N = wkv7.HEAD_SIZE


class CudaSpanSolver:
    """The span computations on this rank's GPU, through the C ABI.  With
    ``nseg`` = 1 the summaries M, Z and D come from the state passes alone
    (wkv7_forward_state, wkv7_backward_state); ``nseg`` > 1 cuts every
    sequence of the span once more into segments that run side by side (the
    time-split entry points)."""

    def __init__(self, nseg: int = 1):
        self.nseg = nseg

    def span_map(self, x: Dict[str, torch.Tensor]) -> Tuple[torch.Tensor, torch.Tensor]:
        r = x["r"]
        B, T, H, _ = r.shape
        eye = torch.eye(N, device=r.device).expand(B, H, N, N).contiguous()
        if self.nseg == 1:
            M = wkv7.forward_state(x["w"], x["k"], None, x["a"], x["b"], s0=eye)
            Z = wkv7.forward_state(x["w"], x["k"], x["v"], x["a"], x["b"])
            return M, Z
        zero_v = torch.zeros_like(x["v"])
        xs0 = [x[n] if n != "v" else zero_v for n in "rwkvab"]
        _, M, _ = wkv7.forward_timesplit(*xs0, s0=eye, nseg=self.nseg)
        _, Z, _ = wkv7.forward_timesplit(*(x[n] for n in "rwkvab"), s0=None, nseg=self.nseg)
        return M, Z

    def forward(self, x, s0):
        if self.nseg == 1:  # checkpoints and the factor cache for the backward
            y, sT, ck, fac = wkv7.forward(*(x[n] for n in "rwkvab"), s0=s0, L=16, want_factors=True)
            return y, sT, (ck, fac)
        y, sT, ws = wkv7.forward_timesplit(*(x[n] for n in "rwkvab"), s0=s0, nseg=self.nseg)
        return y, sT, ws

    def state_grad(self, x, ctx, dy):
        """D: the gradient the span sends to its start when none arrives at its end."""
        if self.nseg == 1:
            return wkv7.backward_state(x["r"], x["w"], x["a"], x["b"], ctx[1], dy)
        return self.backward(x, ctx, dy, None)["ds0"]

    def backward(self, x, ctx, dy, dsT):
        if self.nseg == 1:
            ck, fac = ctx
            return wkv7.backward(*(x[n] for n in "rwkvab"), ck, dy, dsT=dsT, L=16, factors=fac)
        return wkv7.backward_timesplit(*(x[n] for n in "rwkvab"), dy, dsT=dsT, nseg=self.nseg, workspace=ctx)

    def scan(self, M, C, init, backward):
        return wkv7.segment_scan(M, C, init=init, backward=backward)


def _all_gather_states(t: torch.Tensor, group) -> torch.Tensor:
    """[B][H][N][N] per rank -> [B][world][H][N][N] (rank order) on every rank."""
    world = dist.get_world_size(group)
    via_cpu = dist.get_backend(group) == "gloo" and t.is_cuda
    src = t.cpu() if via_cpu else t.contiguous()
    parts = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(parts, src, group=group)
    out = torch.stack(parts, dim=1).contiguous()
    return out.to(t.device) if via_cpu else out


def forward(x: Dict[str, torch.Tensor], s0: Optional[torch.Tensor] = None, group=None, solver=None):
    """This rank's span of y, the sequences' final state (the same on every
    rank) and a context for ``backward``.  ``x`` holds r, w, k, v, a, b of the
    span; ``s0`` the sequences' initial state (read on every rank)."""
    solver = solver or CudaSpanSolver()
    rank = dist.get_rank(group)
    M, Z = solver.span_map(x)
    Mg, Zg = _all_gather_states(M, group), _all_gather_states(Z, group)
    starts, sT = solver.scan(Mg, Zg, s0, False)
    y, _, ctx = solver.forward(x, starts[:, rank].contiguous())
    return y, sT, {"span": ctx, "M": Mg}


def backward(x: Dict[str, torch.Tensor], ctx, dy: torch.Tensor, dsT: Optional[torch.Tensor] = None, group=None,
             solver=None) -> Dict[str, torch.Tensor]:
    """Gradients of this rank's span (dr, dw, dk, dv, da, db) and the
    sequences' ds0 (the same on every rank); ``dsT`` is read on every rank."""
    solver = solver or CudaSpanSolver()
    rank = dist.get_rank(group)
    D = solver.state_grad(x, ctx["span"], dy)
    Dg = _all_gather_states(D, group)
    ends, ds0 = solver.scan(ctx["M"], Dg, dsT, True)
    g = solver.backward(x, ctx["span"], dy, ends[:, rank].contiguous())
    g["ds0"] = ds0
    return g
