"""wkv7_forward_state / wkv7_backward_state: the end state and the start-state
gradient alone, the summaries a span of a sequence gives the segment scan.

The gradient of the state does not depend on the state, so the backward's
state pass runs only that chain (no checkpoint, no k or v, no per-token
gradient) with the full backward's operations in its order: its ds0 must be
bit-identical to wkv7_backward's, on the factorised chunks and on the
chunks that take the exact per-token path.  The forward's state passes are
checked the same way against wkv7_forward's sT (v = 0 against a zero v)."""
import pytest
import torch

from rwkv_linear_attention_wkv7_gb300 import build, synthetic, wkv7
from tests import parity

pytestmark = pytest.mark.gpu


def _inputs(B, T, H, dtype, seed, s0_std=0.1, with_dsT=True, extreme=False):
    spec = synthetic.WorkloadSpec("state_pass", B, T, H, dtype=dtype, s0_std=s0_std, with_dsT=with_dsT, seed=seed)
    d = synthetic.make_inputs(spec, device="cuda")
    if extreme:  # chunks on the exact per-token path: a zero decay, a run of tiny ones, one small w
        w = d["w"].clone()
        w[0, 20, 0, :] = 0.0
        w[-1, 33:47, H - 1, :7] = 1e-3
        w[0, T - 3, H - 1, 5] = 1e-6
        d["w"] = w
    return d


@pytest.mark.parametrize("B,T,H,dtype,with_dsT,extreme", [
    (2, 96, 3, "bf16", True, False),
    (3, 80, 2, "f32", True, False),
    (2, 77, 2, "bf16", False, False),   # ragged last chunk, no dsT
    (2, 80, 3, "f32", True, True),      # exact per-token chunks
    (2, 80, 3, "bf16", False, True),
    (1, 16, 1, "f32", True, False),     # one chunk
])
def test_backward_state_bit_identical(B, T, H, dtype, with_dsT, extreme):
    build()
    d = _inputs(B, T, H, dtype, seed=41, with_dsT=with_dsT, extreme=extreme)
    xs = [d[n] for n in parity.INPUTS]
    _, _, ck, fac = wkv7.forward(*xs, s0=d["s0"], L=16, want_factors=True)
    ref = wkv7.backward(*xs, ck, d["dy"], dsT=d["dsT"], L=16, factors=fac)["ds0"]
    got = wkv7.backward_state(d["r"], d["w"], d["a"], d["b"], fac, d["dy"], dsT=d["dsT"])
    torch.cuda.synchronize()
    wkv7.async_status()
    assert torch.equal(got, ref)


def test_state_passes_no_tokens():
    """T = 0: ds0 = dsT and sT = s0 (or zeros)."""
    build()
    B, H = 2, 3
    z = torch.empty((B, 0, H, 64), device="cuda")
    fac = torch.empty((B, H, 0), device="cuda")
    dsT = torch.randn((B, H, 64, 64), device="cuda")
    assert torch.equal(wkv7.backward_state(z, z, z, z, fac, z, dsT=dsT), dsT)
    assert torch.equal(wkv7.backward_state(z, z, z, z, fac, z), torch.zeros_like(dsT))
    assert torch.equal(wkv7.forward_state(z, z, z, z, z, s0=dsT), dsT)
    assert torch.equal(wkv7.forward_state(z, z, None, z, z), torch.zeros_like(dsT))


@pytest.mark.parametrize("B,T,H,dtype,extreme", [(2, 96, 3, "bf16", False), (2, 77, 2, "f32", False),
                                                 (2, 80, 3, "f32", True)])
def test_forward_state_bit_identical(B, T, H, dtype, extreme):
    """sT from s0 (v given), and the transition product from I with v read as zero."""
    build()
    d = _inputs(B, T, H, dtype, seed=42, extreme=extreme)
    xs = [d[n] for n in parity.INPUTS]
    _, sT, _ = wkv7.forward(*xs, s0=d["s0"], L=16)
    got = wkv7.forward_state(d["w"], d["k"], d["v"], d["a"], d["b"], s0=d["s0"])
    eye = torch.eye(64, device="cuda").expand(B, H, 64, 64).contiguous()
    zv = [torch.zeros_like(x) if n == "v" else x for n, x in zip(parity.INPUTS, xs)]
    _, M, _ = wkv7.forward(*zv, s0=eye, L=16)
    gotM = wkv7.forward_state(d["w"], d["k"], None, d["a"], d["b"], s0=eye)
    torch.cuda.synchronize()
    wkv7.async_status()
    assert torch.equal(got, sT)
    assert torch.equal(gotM, M)


def test_span_summaries_join_through_the_scan():
    """Two spans of one sequence joined by wkv7_segment_scan give the
    whole-sequence sT and ds0 within the parity bars: the summaries are the
    state passes' M, Z (forward) and D (backward)."""
    build()
    d = _inputs(2, 128, 2, "bf16", seed=43)
    xs = [d[n] for n in parity.INPUTS]
    B, T, H, N = d["r"].shape
    half = T // 2
    spans = [[x[:, s * half:(s + 1) * half].contiguous() for x in xs] for s in range(2)]
    dys = [d["dy"][:, s * half:(s + 1) * half].contiguous() for s in range(2)]
    eye = torch.eye(N, device="cuda").expand(B, H, N, N).contiguous()
    M = torch.stack([wkv7.forward_state(x[1], x[2], None, x[4], x[5], s0=eye) for x in spans], 1).contiguous()
    Z = torch.stack([wkv7.forward_state(x[1], x[2], x[3], x[4], x[5]) for x in spans], 1).contiguous()
    starts, sT = wkv7.segment_scan(M, Z, init=d["s0"])
    facs = [wkv7.forward(*x, s0=starts[:, s].contiguous(), L=16, want_factors=True)[3] for s, x in enumerate(spans)]
    D = torch.stack([wkv7.backward_state(x[0], x[1], x[4], x[5], f, dy) for x, f, dy in zip(spans, facs, dys)],
                    1).contiguous()
    _, ds0 = wkv7.segment_scan(M, D, init=d["dsT"], backward=True)
    _, sT_ref, ck, fac = wkv7.forward(*xs, s0=d["s0"], L=16, want_factors=True)
    ds0_ref = wkv7.backward(*xs, ck, d["dy"], dsT=d["dsT"], L=16, factors=fac)["ds0"]
    torch.cuda.synchronize()
    wkv7.async_status()
    assert parity.max_rel(sT.double().cpu().numpy(), sT_ref.double().cpu().numpy()) <= parity.FWD_TOL
    assert parity.max_rel(ds0.double().cpu().numpy(), ds0_ref.double().cpu().numpy()) <= 1e-3
