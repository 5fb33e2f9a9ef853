"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from rwkv_linear_attention_wkv7_gb300 import synthetic, wkv7
from tests import parity

pytestmark = pytest.mark.gpu

SMALL = ["tiny_b1_t64_h4", "stream_b1_t512_h48", "mid_b8_t1024_h12"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from rwkv_linear_attention_wkv7_gb300 import build
    build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", SMALL)
def test_small_workloads_all_heads(name):
    """Every head of the small workloads: forward (y, sT, checkpoints) and all gradients."""
    spec = synthetic.WORKLOADS[name]
    d, host = parity.inputs_on_device(spec)
    out = parity.run_gpu(d, L=spec.L)
    worst = parity.check_heads(host, out, parity.all_heads(spec.B, spec.H), L=spec.L)
    print(name, {k: f"{v:.2e}" for k, v in worst.items()})


def _custom(B, T, H, dtype="f32", s0_std=0.1, dsT=True, seed=3, w_shift=0.0):
    return synthetic.WorkloadSpec("custom", B, T, H, dtype=dtype, s0_std=s0_std, with_dsT=dsT, seed=seed,
                                  w_shift=w_shift)


@pytest.mark.parametrize("T,L", [(1, 16), (15, 16), (17, 16), (37, 5), (37, 1), (100, 64), (130, 16), (45, 200)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_lengths_and_strides(T, L, dtype):
    """Ragged sequence lengths (partial staging chunks, partial checkpoint
    intervals, partial backward windows) with an initial state and dsT."""
    spec = _custom(2, T, 3, dtype=dtype)
    d, host = parity.inputs_on_device(spec)
    out = parity.run_gpu(d, L=L)
    assert out["ckpt"].shape[2] == (T + L - 1) // L
    parity.check_heads(host, out, parity.all_heads(2, 3), L=L)


@pytest.mark.parametrize("T", [15, 130, 512])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_with_and_without_factor_cache(T, dtype):
    """The backward that reuses the forward's per-chunk factors and the one
    that recomputes them both match the oracle, and agree with each other to
    fp32 rounding."""
    spec = _custom(2, T, 3, dtype=dtype)
    d, host = parity.inputs_on_device(spec)
    with_fac = parity.run_gpu(d, L=16, factors=True)
    without = parity.run_gpu(d, L=16, factors=False)
    heads = parity.all_heads(2, 3)
    parity.check_heads(host, with_fac, heads, L=16)
    parity.check_heads(host, without, heads, L=16)
    for k in parity.GRADS + ("ds0",):  # different kernels, same split products in another order
        a, b = with_fac[k].double(), without[k].double()
        assert float((a - b).abs().max() / b.abs().max().clamp_min(1e-30)) <= 1e-4, k


@pytest.mark.parametrize("T", [16, 130, 512])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tensor_core_and_warp_mma_backward(T, dtype, monkeypatch):
    """The backward with the factor cache, with two of its 64-row state
    products on tcgen05 (selected by WKV7_BACKWARD_KERNEL=tcgen05) and all on
    warp-level mma.sync (the default): the same split products in another
    order.  Both match the oracle element by element, and each other to fp32
    rounding (1e-4 of the largest element: dw, a running sum over the chunk,
    collects the most of it)."""
    spec = _custom(2, T, 3, dtype=dtype, seed=13)
    d, host = parity.inputs_on_device(spec)
    mma = parity.run_gpu(d, L=16, factors=True)
    monkeypatch.setenv("WKV7_BACKWARD_KERNEL", "tcgen05")
    tc = parity.run_gpu(d, L=16, factors=True)
    monkeypatch.delenv("WKV7_BACKWARD_KERNEL")
    heads = parity.all_heads(2, 3)
    parity.check_heads(host, tc, heads, L=16)
    parity.check_heads(host, mma, heads, L=16)
    for k in parity.GRADS + ("ds0",):
        a, b = tc[k].double(), mma[k].double()
        assert float((a - b).abs().max() / b.abs().max().clamp_min(1e-30)) <= 1e-4, k


def test_empty_sequence():
    """T = 0: the forward copies s0 to sT, the backward copies dsT to ds0."""
    B, H, N = 2, 3, 64
    s0 = torch.randn(B, H, N, N, device="cuda")
    dsT = torch.randn(B, H, N, N, device="cuda")
    e = torch.empty(B, 0, H, N, device="cuda")
    y, sT, ck, fac = wkv7.forward(e, e, e, e, e, e, s0=s0, L=16, want_factors=True)
    assert y.shape == (B, 0, H, N) and ck.shape == (B, H, 0, N, N) and fac.shape == (B, H, 0)
    assert torch.equal(sT, s0)
    g = wkv7.backward(e, e, e, e, e, e, ck, torch.empty(B, 0, H, N, device="cuda"), dsT=dsT, L=16, factors=fac)
    assert torch.equal(g["ds0"], dsT)
    _, sT0, _ = wkv7.forward(e, e, e, e, e, e, s0=None, L=16)
    torch.cuda.synchronize()
    assert torch.count_nonzero(sT0) == 0


def test_bitwise_reproducible():
    """Two runs on the same inputs give bit-identical y, sT, checkpoints and gradients."""
    d, _ = parity.inputs_on_device(_custom(2, 200, 4, dtype="bf16"))
    o1 = parity.run_gpu(d)
    o2 = parity.run_gpu(d)
    for k in o1:
        if o1[k] is not None:
            assert torch.equal(o1[k], o2[k]), k


def test_decode_step_from_nonzero_state():
    """One decode token from the state a T=512 forward (nonzero s0) ends in --
    the streaming-inference case -- against the oracle's decode step."""
    spec = synthetic.WORKLOADS["stream_b1_t512_h48"]
    d, _ = parity.inputs_on_device(spec)
    out = parity.run_gpu(d, backward=False)
    tok = synthetic.make_inputs(synthetic.WorkloadSpec("token", 1, 1, spec.H, seed=12))
    vec = {n: tok[n][:, 0].contiguous() for n in parity.INPUTS}
    host_state = out["sT"].cpu()
    state = out["sT"].clone()
    y = wkv7.decode_step(*(vec[n].cuda() for n in parity.INPUTS), state)
    torch.cuda.synchronize()
    ry, rs = oracle.decode_step(*(vec[n] for n in parity.INPUTS), host_state)
    assert parity.max_rel(y.cpu().double().numpy(), ry) <= parity.FWD_TOL
    assert parity.max_rel(state.cpu().double().numpy(), rs) <= parity.FWD_TOL


def test_decode_chain_matches_forward():
    """Feeding tokens one by one through the decode step reproduces the
    sequence forward (bf16 inputs), within the forward tolerance (the
    sequence forward sums in a different order than the per-token step)."""
    spec = _custom(2, 24, 5, dtype="bf16")
    d, _ = parity.inputs_on_device(spec)
    out = parity.run_gpu(d, backward=False)
    state = d["s0"].clone()
    ys = [wkv7.decode_step(*(d[n][:, t].contiguous() for n in parity.INPUTS), state) for t in range(spec.T)]
    y = torch.stack(ys, 1)
    torch.cuda.synchronize()
    assert parity.max_rel(y.double().cpu().numpy(), out["y"].double().cpu().numpy()) <= parity.FWD_TOL
    assert parity.max_rel(state.double().cpu().numpy(), out["sT"].double().cpu().numpy()) <= parity.FWD_TOL


def test_batched_decode_workload_sampled_heads():
    """The batched streaming-decode workload at its full size (B=512
    sequences, H=32, bf16 vectors, carried state): three chained decode calls
    in the launch configuration the benchmark times, then sampled heads
    against the oracle's decode step applied three times to the same head."""
    spec = synthetic.DECODE_WORKLOADS["decode_b512_h32"]
    d = synthetic.make_inputs(spec)
    state = d["s0"].cuda()
    y = torch.empty((spec.B, spec.H, spec.N), device="cuda")
    ys = []
    for t in range(3):
        wkv7.decode_step(*(d[n][:, t].contiguous().cuda() for n in parity.INPUTS), state, y=y)
        ys.append(y.cpu())
    torch.cuda.synchronize()
    g = np.random.default_rng(5)
    for _ in range(12):
        b, h = int(g.integers(0, spec.B)), int(g.integers(0, spec.H))
        hs = d["s0"][b:b + 1, h:h + 1].clone()
        for t in range(3):
            vec = [d[n][b:b + 1, t, h:h + 1].contiguous() for n in parity.INPUTS]
            ry, hs = oracle.decode_step(*vec, hs)  # the oracle carries its state in fp64
            assert parity.max_rel(ys[t][b:b + 1, h:h + 1].double().numpy(), ry) <= parity.FWD_TOL
        assert parity.max_rel(state[b:b + 1, h:h + 1].cpu().double().numpy(), hs) <= parity.FWD_TOL


def test_autograd_function():
    """The torch.autograd wrapper routes gradients from the library."""
    spec = _custom(1, 33, 2)
    d, host = parity.inputs_on_device(spec)
    xs = [d[n].clone().requires_grad_(True) for n in parity.INPUTS]
    s0 = d["s0"].clone().requires_grad_(True)
    y, sT = wkv7.wkv7(*xs, s0=s0, L=16)
    ((y * d["dy"]).sum() + (sT * d["dsT"]).sum()).backward()
    ref = parity.oracle_head(host, 0, 1, L=16)
    for n, x in zip(parity.GRADS, xs):
        assert parity.grad_rel(x.grad[:, :, 1:2].double().cpu().numpy(), ref[n]) <= parity.GRAD_TOL, n
    assert parity.grad_rel(s0.grad[:, 1:2].double().cpu().numpy(), ref["ds0"]) <= parity.GRAD_TOL


@pytest.mark.slow
@pytest.mark.parametrize("name", ["bf16_b16_t4096_h32", "long_b64_t4096_h40"])
def test_full_size_sampled_heads(name):
    """The full-size workloads, run in the launch configuration the bench
    times, checked on sampled heads the oracle recomputes over all T."""
    spec = synthetic.WORKLOADS[name]
    heads = parity.sample_heads(spec.B, spec.H, n=6)
    d, host = parity.inputs_on_device(spec, heads=heads)
    out = parity.run_gpu(d, L=spec.L)
    for k in ("y", "sT") + parity.GRADS + ("ds0",):
        assert bool(torch.isfinite(out[k]).all()), k
    worst = parity.check_heads(host, out, heads, L=spec.L)
    print(name, {k: f"{v:.2e}" for k, v in worst.items()})


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_decay_chunks(dtype):
    """Chunks whose cumulative decay underflows (w = 0 for a token, or a run of
    tiny w) next to ordinary chunks: the forward takes the exact per-token
    path there and must still match the oracle."""
    spec = _custom(2, 80, 3, dtype=dtype)
    d, host = parity.inputs_on_device(spec)
    for x in (d, host):
        w = x["w"].clone()
        w[0, 20, 0, :] = 0.0               # hard reset of head 0 in chunk 1
        w[1, 33:47, 1, :7] = 1e-3          # long run of tiny decay in chunk 2 of head (1,1)
        w[0, 70, 2, 5] = 0.0               # a single zero column in the last chunk
        x["w"] = w.to(x["w"].device) if x is d else w
    out = parity.run_gpu(d, L=16)
    parity.check_heads(host, out, parity.all_heads(2, 3), L=16)


@pytest.mark.parametrize("wv", [1e-2, 1e-4, 1e-6])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_isolated_small_decays(wv, dtype):
    """Single tokens (and one partial key range) with a small decay w inside
    otherwise ordinary chunks: the cumulative decay stays far inside the range
    the factorised form accepts, so only the backward's small-w rule keeps dw
    exact there (dw is recovered from w o dw by a division by w).  Every
    gradient is checked element by element."""
    spec = _custom(2, 80, 3, dtype=dtype, seed=7)
    d, host = parity.inputs_on_device(spec)
    for x in (d, host):
        w = x["w"].clone()
        w[0, 5, 0, :] = wv           # chunk 0, one token, every key
        w[0, 40, 1, :] = wv          # chunk 2
        w[1, 63, 2, :] = wv          # last token of chunk 3
        w[1, 17, 0, 10:30] = wv      # some keys of one token
        x["w"] = w.to(x["w"].device)
    out = parity.run_gpu(d, L=16)
    parity.check_heads(host, out, parity.all_heads(2, 3), L=16)


def test_forward_paths_agree():
    """Checkpoint strides that are multiples of 16 run the chunked tensor-core
    forward; others run the per-token kernel.  Both give the same y and sT."""
    spec = _custom(2, 100, 4, dtype="bf16")
    d, _ = parity.inputs_on_device(spec)
    y1, s1, _ = wkv7.forward(*(d[n] for n in parity.INPUTS), s0=d["s0"], L=16)
    y2, s2, _ = wkv7.forward(*(d[n] for n in parity.INPUTS), s0=d["s0"], L=7)
    torch.cuda.synchronize()
    assert parity.max_rel(y1.double().cpu().numpy(), y2.double().cpu().numpy()) <= parity.FWD_TOL
    assert parity.max_rel(s1.double().cpu().numpy(), s2.double().cpu().numpy()) <= parity.FWD_TOL


# ---- the producers fused into the entry points (w_pre, kk, avec in; dw_pre, dkk, davec out)

@pytest.mark.parametrize("name", SMALL)
def test_fused_small_workloads_all_heads(name):
    """Every head of the small workloads through the fused entry points:
    forward (y, sT, checkpoints) and the gradients of the fused inputs."""
    spec = synthetic.WORKLOADS[name]
    d, host = parity.inputs_on_device(spec, fused=True)
    out = parity.run_gpu(d, L=16, fused=True)
    worst = parity.check_heads(host, out, parity.all_heads(spec.B, spec.H), L=16, fused=True)
    print(name, {k: f"{v:.2e}" for k, v in worst.items()})


@pytest.mark.parametrize("T", [1, 15, 17, 130])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_ragged_lengths(T, dtype):
    """Ragged lengths (partial chunks) with an initial state and dsT, fused path;
    a saturating decay pre-activation shift exercises w near exp(-0.606531)."""
    spec = synthetic.WorkloadSpec("custom", 2, T, 3, dtype=dtype, s0_std=0.1, with_dsT=True, seed=4, w_shift=2.0)
    d, host = parity.inputs_on_device(spec, fused=True)
    out = parity.run_gpu(d, L=16, fused=True)
    parity.check_heads(host, out, parity.all_heads(2, 3), L=16, fused=True)


@pytest.mark.parametrize("w_shift", [-3.0, -10.0])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_negative_decay_shift(w_shift, dtype):
    """Decay pre-activations shifted down (w close to 1, as in the long fp32
    workload's distribution at -3 and far beyond it at -10): dw_pre needs the
    sigmoid's own relative precision where the sigmoid is tiny."""
    spec = synthetic.WorkloadSpec("custom", 2, 130, 3, dtype=dtype, s0_std=0.1, with_dsT=True, seed=4,
                                  w_shift=w_shift)
    d, host = parity.inputs_on_device(spec, fused=True)
    out = parity.run_gpu(d, L=16, fused=True)
    parity.check_heads(host, out, parity.all_heads(2, 3), L=16, fused=True)


def test_fused_forward_longer_stride():
    """The fused forward with checkpoint stride 32 (a multiple of the chunk)."""
    spec = synthetic.WorkloadSpec("custom", 1, 100, 2, s0_std=0.1, seed=6)
    d, host = parity.inputs_on_device(spec, fused=True)
    out = parity.run_gpu(d, L=32, backward=False, factors=False, fused=True)
    assert out["ckpt"].shape[2] == 4
    parity.check_heads(host, out, parity.all_heads(1, 2), L=32, backward=False, fused=True)


@pytest.mark.slow
def test_fused_full_size_sampled_heads():
    """The fused entry points on the full-size bf16 workload (B=16, T=4096,
    H=32), sampled heads recomputed by the oracle over all T."""
    spec = synthetic.WORKLOADS["bf16_b16_t4096_h32"]
    heads = parity.sample_heads(spec.B, spec.H, n=4)
    d, host = parity.inputs_on_device(spec, heads=heads, fused=True)
    out = parity.run_gpu(d, L=16, fused=True)
    for k in ("y", "sT") + parity.GRADS_FUSED + ("ds0",):
        assert bool(torch.isfinite(out[k]).all()), k
    parity.check_heads(host, out, heads, L=16, fused=True)


# ---- the GroupNorm + bonus output epilogue fused into the recurrence

def _gn_case(spec, seed=5):
    d, host = parity.inputs_on_device(spec)
    gp = synthetic.gn_params(spec.H, seed=seed)
    return d, host, gp, {n: t.cuda() for n, t in gp.items()}


@pytest.mark.parametrize("name", ["tiny_b1_t64_h4", "mid_b8_t1024_h12"])
def test_gn_epilogue_all_heads(name):
    """Recurrence + GroupNorm + bonus against the oracle composite on every
    head: o, y, sT, checkpoints, the seven gradients (dr, dk, dv with the
    bonus's own terms) and the parameter gradients summed over batch rows."""
    spec = synthetic.WORKLOADS[name]
    d, host, gp, gpd = _gn_case(spec)
    out = parity.run_gpu_gn(d, gpd)
    worst = parity.check_heads_gn(host, gp, out, parity.all_heads(spec.B, spec.H), spec.B)
    print(name, {k: f"{v:.2e}" for k, v in worst.items()})


@pytest.mark.parametrize("T", [1, 15, 17, 130])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gn_epilogue_ragged(T, dtype):
    """Ragged lengths (padding tokens of the last chunk must not reach the
    parameter sums), with an initial state and dsT."""
    spec = _custom(2, T, 3, dtype=dtype, seed=17)
    d, host, gp, gpd = _gn_case(spec, seed=6)
    out = parity.run_gpu_gn(d, gpd)
    parity.check_heads_gn(host, gp, out, parity.all_heads(2, 3), 2)


def test_gn_epilogue_extreme_decay_chunk():
    """A chunk on the exact per-token path (w = 0 for a token) adds the
    bonus's terms there too."""
    spec = _custom(2, 48, 2, dtype="bf16", seed=18)
    d, host, gp, gpd = _gn_case(spec, seed=7)
    for x in (d, host):
        w = x["w"].clone()
        w[1, 20, 0, :] = 0.0
        x["w"] = w.to(x["w"].device)
    out = parity.run_gpu_gn(d, gpd)
    parity.check_heads_gn(host, gp, out, parity.all_heads(2, 2), 2)


@pytest.mark.slow
def test_gn_epilogue_full_size():
    """The bf16 B=16 T=4096 H=32 workload through the epilogue entry points:
    two head indices over all 16 batch rows (per-token tensors and the
    parameter sums of those heads)."""
    spec = synthetic.WORKLOADS["bf16_b16_t4096_h32"]
    heads = [(b, h) for h in (0, 31) for b in range(spec.B)]
    d, host = parity.inputs_on_device(spec, heads=heads)
    gp = synthetic.gn_params(spec.H, seed=8)
    out = parity.run_gpu_gn(d, {n: t.cuda() for n, t in gp.items()})
    for k in ("o", "y") + parity.GRADS + parity.GN_GRADS:
        assert bool(torch.isfinite(out[k]).all()), k
    worst = parity.check_heads_gn(host, gp, out, heads, spec.B)
    print({k: f"{v:.2e}" for k, v in worst.items()})
