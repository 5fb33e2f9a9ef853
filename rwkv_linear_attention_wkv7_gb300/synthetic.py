"""Seeded synthetic WKV7 inputs, shared by the CUDA-side tests/bench and the oracle.

This module only draws random numbers and shapes them into the inputs the
WKV7 recurrence is fed in an RWKV-7 time-mix block; it holds none of the
recurrence's arithmetic.  The shaping follows the producers of the
"Foundry/cuda_kernels/timemix.cu" page:

* k_l2norm: kk = x / (||x||_2 + 1e-12) per (b, t, h) over the head's N lanes;
* k_composites: the kernel's composite vectors are a = -kk, b = kk * gate,
  with gate = sigmoid(.) (k_bias_sigmoid);
* k_decay: w = exp(-0.606531 * sigmoid(.)), 0.606531 = e^{-1/2}.

Draw order (one torch CPU generator, fp32 N(0,1) unless stated):
r, k, v, kk_raw, gate_raw, w_raw (+ w_shift), s0 (x s0_std), dy, dsT.
Every tensor is drawn even when unused, so the stream is the same for every
option set.  For ``dtype='bf16'`` the six recurrence inputs are rounded to
bf16 after shaping; s0, dy, dsT stay fp32.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Iterator, Optional, Tuple

import torch

DECAY_COEFF = 0.606531  # e^{-1/2}, the decay scale of the timemix page's k_decay


@dataclass(frozen=True)
class WorkloadSpec:
    """One WKV7 workload: sizes, input distributions and checkpoint stride."""
    name: str
    B: int
    T: int
    H: int
    N: int = 64
    dtype: str = "f32"          # dtype of r, w, k, v, a, b: "f32" or "bf16"
    s0_std: float = 0.0         # 0 -> zero initial state
    w_shift: float = 0.0        # mean of the decay pre-activation
    with_dsT: bool = False      # draw a final-state gradient
    L: int = 16                 # checkpoint stride (tokens)
    seed: int = 0

    @property
    def elems(self) -> int:
        return self.B * self.T * self.H * self.N

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five workloads this library is tested and measured on, named by size.
WORKLOADS: Dict[str, WorkloadSpec] = {
    "tiny_b1_t64_h4": WorkloadSpec("tiny_b1_t64_h4", 1, 64, 4),
    "stream_b1_t512_h48": WorkloadSpec("stream_b1_t512_h48", 1, 512, 48, s0_std=0.1),
    "mid_b8_t1024_h12": WorkloadSpec("mid_b8_t1024_h12", 8, 1024, 12),
    "bf16_b16_t4096_h32": WorkloadSpec("bf16_b16_t4096_h32", 16, 4096, 32, dtype="bf16"),
    "long_b64_t4096_h40": WorkloadSpec("long_b64_t4096_h40", 64, 4096, 40, s0_std=0.1,
                                       w_shift=-3.0, with_dsT=True),
}

# Batched streaming decode: many sequences advance one token per call from a
# carried state.  T here is the number of distinct token sets drawn (a decode
# run cycles through them); s0 is the carried state.
DECODE_WORKLOADS: Dict[str, WorkloadSpec] = {
    "decode_b512_h32": WorkloadSpec("decode_b512_h32", 512, 8, 32, dtype="bf16", s0_std=0.1),
}

# Few, long sequences: B*H = 8 heads of 65536 tokens (the time-split entry
# points' case: one thread block per head would leave the GPU nearly idle).
TIMESPLIT_WORKLOADS: Dict[str, WorkloadSpec] = {
    "long_b1_t65536_h8": WorkloadSpec("long_b1_t65536_h8", 1, 65536, 8, dtype="bf16", s0_std=0.1, with_dsT=True),
}


def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def stream_inputs(spec: WorkloadSpec, fused: bool = False) -> Iterator[Tuple[str, Optional[torch.Tensor]]]:
    """Yield (name, CPU tensor) in a fixed order, holding few tensors at once.

    Names: r, k, v, a, b, w, s0, dy, dsT (s0 / dsT may be None).  With
    ``fused`` the same draws come out before the producers: kk, avec and
    w_pre in place of a, b and w (the inputs of the fused entry points).
    """
    g = torch.Generator().manual_seed(spec.seed)
    shape = (spec.B, spec.T, spec.H, spec.N)
    sshape = (spec.B, spec.H, spec.N, spec.N)
    dt = _torch_dtype(spec.dtype)

    def cast(x):
        return x.to(dt) if dt != torch.float32 else x

    yield "r", cast(torch.randn(shape, generator=g))
    yield "k", cast(torch.randn(shape, generator=g))
    yield "v", cast(torch.randn(shape, generator=g))
    kk = torch.randn(shape, generator=g)
    kk = kk / (kk.norm(dim=-1, keepdim=True) + 1e-12)
    gate = torch.sigmoid(torch.randn(shape, generator=g))
    if fused:
        yield "kk", cast(kk)
        yield "avec", cast(gate)
    else:
        yield "a", cast(-kk)
        yield "b", cast(kk * gate)
    del kk, gate
    w_raw = torch.randn(shape, generator=g)
    if spec.w_shift:
        w_raw += spec.w_shift
    if fused:
        yield "w_pre", cast(w_raw)
    else:
        yield "w", cast(torch.exp(-DECAY_COEFF * torch.sigmoid(w_raw)))
    del w_raw
    s0 = torch.randn(sshape, generator=g) * spec.s0_std
    yield "s0", s0 if spec.s0_std > 0 else None
    yield "dy", torch.randn(shape, generator=g)
    dsT = torch.randn(sshape, generator=g)
    yield "dsT", dsT if spec.with_dsT else None


def gn_params(H: int, N: int = 64, seed: int = 0) -> Dict[str, torch.Tensor]:
    """Seeded weights of the GroupNorm + bonus output epilogue, each [H][N]
    fp32 (one generator, draw order gn_w, gn_b, r_k): gn_w = 1 + 0.5 N(0,1),
    gn_b = 0.5 N(0,1), r_k = 0.5 N(0,1) -- trained-looking scales around the
    identity GroupNorm, with no trained values involved."""
    g = torch.Generator().manual_seed(seed)
    gn_w = 1.0 + 0.5 * torch.randn((H, N), generator=g)
    gn_b = 0.5 * torch.randn((H, N), generator=g)
    r_k = 0.5 * torch.randn((H, N), generator=g)
    return {"gn_w": gn_w, "gn_b": gn_b, "r_k": r_k}


def make_inputs(spec: WorkloadSpec, device: str = "cpu", fused: bool = False) -> Dict[str, Optional[torch.Tensor]]:
    """All inputs of ``spec`` as a dict, moved to ``device`` one by one."""
    out = {}
    for name, t in stream_inputs(spec, fused=fused):
        out[name] = None if t is None else t.to(device)
    return out


def head_slice(x: Optional[torch.Tensor], b: int, h: int, state: bool = False):
    """The (b, h) sub-problem of a [B][T][H][N] (or [B][H][N][N]) tensor, as B=H=1."""
    if x is None:
        return None
    if state:
        return x[b:b + 1, h:h + 1].contiguous()
    return x[b:b + 1, :, h:h + 1, :].contiguous()
