"""wkv7_forward_backward: one training step (forward with checkpoints and the
factor cache, then the backward) run as concurrent blocks of batch rows on the
library's own streams.

Every output must be bit-identical to wkv7_forward followed by wkv7_backward
on the whole batch: the blocks launch the same kernels on row slices, and the
heads of different rows never meet.  One case is also checked head by head
against the oracle."""
import dataclasses

import pytest
import torch

from rwkv_linear_attention_wkv7_gb300 import build, synthetic, wkv7
from tests import parity

pytestmark = pytest.mark.gpu

OUTS = ("y", "sT", "ckpt") + parity.GRADS + ("ds0",)


def _separate(d, want_factors):
    res = wkv7.forward(*(d[n] for n in parity.INPUTS), s0=d["s0"], L=16, want_factors=want_factors)
    out = {"y": res[0], "sT": res[1], "ckpt": res[2], "factors": res[3] if want_factors else None}
    out.update(wkv7.backward(*(d[n] for n in parity.INPUTS), res[2], d["dy"], dsT=d["dsT"], L=16,
                             factors=out["factors"]))
    return out


@pytest.mark.parametrize("B,T,H,dtype,s0_std,with_dsT,nsplit,want_factors", [
    (4, 200, 3, "bf16", 0.1, True, 0, True),   # the default split, ragged T
    (3, 64, 2, "f32", 0.0, True, 2, True),     # blocks of 1 and 2 rows
    (5, 48, 2, "bf16", 0.1, False, 4, True),   # four blocks of unequal size
    (2, 33, 4, "f32", 0.1, True, 3, True),     # more blocks than rows: one row each
    (3, 40, 2, "bf16", 0.1, True, 2, False),   # no factor cache: the backward rebuilds it
    (1, 32, 2, "f32", 0.1, True, 0, True),     # one row: the two calls in order
    (2, 0, 2, "f32", 0.1, True, 2, True),      # T = 0: sT = s0, ds0 = dsT
])
def test_bit_identical_to_the_two_calls(B, T, H, dtype, s0_std, with_dsT, nsplit, want_factors):
    build()
    spec = synthetic.WorkloadSpec("fwdbwd", B, T, H, dtype=dtype, s0_std=s0_std, with_dsT=with_dsT, seed=31)
    d = synthetic.make_inputs(spec, device="cuda")
    ref = _separate(d, want_factors)
    got = wkv7.forward_backward(*(d[n] for n in parity.INPUTS), d["dy"], s0=d["s0"], dsT=d["dsT"],
                                want_factors=want_factors, nsplit=nsplit)
    torch.cuda.synchronize()
    wkv7.async_status()
    names = OUTS + (("factors",) if want_factors else ())
    for n in names:
        assert torch.equal(got[n], ref[n]), n


def test_against_the_oracle():
    """The default split on every head of a small bf16 workload, element by
    element at the forward and gradient bars."""
    build()
    spec = synthetic.WorkloadSpec("fwdbwd_oracle", 3, 96, 2, dtype="bf16", s0_std=0.1, with_dsT=True, seed=32)
    d, host = parity.inputs_on_device(spec)
    got = wkv7.forward_backward(*(d[n] for n in parity.INPUTS), d["dy"], s0=d["s0"], dsT=d["dsT"])
    torch.cuda.synchronize()
    wkv7.async_status()
    parity.check_heads(host, {k: got[k] for k in OUTS}, parity.all_heads(spec.B, spec.H), L=16)


def test_follows_the_callers_stream():
    """Work queued on the caller's stream before the call is seen by it, and
    work queued after it sees its results: the call's own streams are forked
    from the caller's and joined back into it."""
    build()
    spec = synthetic.WorkloadSpec("fwdbwd_stream", 4, 64, 2, dtype="bf16", s0_std=0.1, with_dsT=True, seed=33)
    d = synthetic.make_inputs(spec, device="cuda")
    ref = _separate(d, True)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        dy = torch.zeros_like(d["dy"])
        torch.cuda._sleep(20_000_000)  # keep the stream busy before dy is filled
        dy.copy_(d["dy"])
        got = wkv7.forward_backward(*(d[n] for n in parity.INPUTS), dy, s0=d["s0"], dsT=d["dsT"], stream=st)
        dr = got["dr"].clone()  # queued after the call on the same stream
    st.synchronize()
    wkv7.async_status()
    assert torch.equal(dr, ref["dr"])


@pytest.mark.parametrize("B,T,H,dtype,nsplit", [(4, 200, 3, "bf16", 0), (3, 48, 2, "f32", 3), (1, 32, 2, "bf16", 2)])
def test_fused_bit_identical_to_the_two_fused_calls(B, T, H, dtype, nsplit):
    """wkv7_forward_backward_fused against wkv7_forward_fused + wkv7_backward_fused."""
    build()
    spec = synthetic.WorkloadSpec("fwdbwd_fused", B, T, H, dtype=dtype, s0_std=0.1, with_dsT=True, seed=34)
    d = synthetic.make_inputs(spec, device="cuda", fused=True)
    ref = parity.run_gpu(d, L=16, fused=True)
    got = wkv7.forward_backward_fused(*(d[n] for n in parity.INPUTS_FUSED), d["dy"], s0=d["s0"], dsT=d["dsT"],
                                      nsplit=nsplit)
    torch.cuda.synchronize()
    wkv7.async_status()
    for n in ("y", "sT", "ckpt") + parity.GRADS_FUSED + ("ds0",):
        assert torch.equal(got[n], ref[n]), n


@pytest.mark.parametrize("B,T,H,dtype,nsplit", [(4, 200, 3, "bf16", 0), (5, 48, 2, "f32", 4), (2, 0, 2, "f32", 2),
                                                (1, 32, 2, "bf16", 2)])
def test_gn_bit_identical_to_the_two_gn_calls(B, T, H, dtype, nsplit):
    """wkv7_forward_backward_gn against wkv7_forward_gn + wkv7_backward_gn: the blocks
    leave their rows' parameter-gradient sums, one reduction over all rows follows
    in the same order, so dgn_w, dgn_b, dr_k are bit-identical too."""
    build()
    spec = synthetic.WorkloadSpec("fwdbwd_gn", B, T, H, dtype=dtype, s0_std=0.1, with_dsT=True, seed=35)
    d = synthetic.make_inputs(spec, device="cuda")
    gp = {n: t.cuda() for n, t in synthetic.gn_params(H, seed=36).items()}
    ref = parity.run_gpu_gn(d, gp)
    got = wkv7.forward_backward_gn(*(d[n] for n in parity.INPUTS), d["dy"], gp["gn_w"], gp["gn_b"], gp["r_k"],
                                   s0=d["s0"], dsT=d["dsT"], nsplit=nsplit)
    torch.cuda.synchronize()
    wkv7.async_status()
    for n in ("o", "y", "sT", "ckpt") + parity.GRADS + ("ds0", "dgn_w", "dgn_b", "dr_k"):
        assert torch.equal(got[n], ref[n]), n


@pytest.mark.parametrize("nsplit", [0, 4])
def test_captured_in_a_cuda_graph(nsplit):
    """The one-call step captures into a CUDA graph (its fork onto the library's
    streams and the join back are ordinary cross-stream captures) and the graph
    replays it: new inputs copied into the captured buffers give the same
    outputs, bit for bit, as the eager call (two and four blocks)."""
    build()
    spec = synthetic.WorkloadSpec("fwdbwd_graph", 4, 96, 2, dtype="bf16", s0_std=0.1, with_dsT=True, seed=37)
    d = synthetic.make_inputs(spec, device="cuda")
    d2 = synthetic.make_inputs(dataclasses.replace(spec, seed=38), device="cuda")
    xs = [d[n].clone() for n in parity.INPUTS]
    dy = d["dy"].clone()
    # warm up outside the capture (the library's streams and device tables exist afterwards)
    out = wkv7.forward_backward(*xs, dy, s0=d["s0"], dsT=d["dsT"], nsplit=nsplit)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        wkv7.forward_backward(*xs, dy, s0=d["s0"], dsT=d["dsT"], nsplit=nsplit, out=out,
                              stream=torch.cuda.current_stream())
    for x, n in zip(xs, parity.INPUTS):
        x.copy_(d2[n])
    dy.copy_(d2["dy"])
    graph.replay()
    torch.cuda.synchronize()
    wkv7.async_status()
    ref = wkv7.forward_backward(*(d2[n] for n in parity.INPUTS), d2["dy"], s0=d["s0"], dsT=d["dsT"], nsplit=1)
    torch.cuda.synchronize()
    for n in OUTS:
        assert torch.equal(out[n], ref[n]), n
