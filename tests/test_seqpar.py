"""Sequence parallelism across ranks (each rank one span of the T axis):
world sizes 2 and 3 on the gloo backend.  On the CPU the span computations are done
by the oracle (a stand-in with the solver interface), which checks the
exchange itself; on the GPU both ranks run the library's kernels on cuda:0
(two processes, exchanging only through gloo between launches).  Either way
each rank's span and the shared sT / ds0 must match the oracle run over the
whole sequence."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

N = 64


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleSpanSolver:
    """Test stand-in for the span computations: the float64 oracle."""

    def span_map(self, x):
        import oracle
        B, T, H, _ = x["r"].shape
        eye = np.broadcast_to(np.eye(N), (B, H, N, N)).copy()
        xs0 = [x[n] if n != "v" else torch.zeros_like(x["v"]) for n in "rwkvab"]
        _, M, _ = oracle.forward(*xs0, s0=eye, L=16, want_ckpt=False)
        _, Z, _ = oracle.forward(*(x[n] for n in "rwkvab"), L=16, want_ckpt=False)
        return torch.from_numpy(M), torch.from_numpy(Z)

    def forward(self, x, s0):
        import oracle
        y, sT, _ = oracle.forward(*(x[n] for n in "rwkvab"), s0=s0, L=16, want_ckpt=False)
        return torch.from_numpy(y), torch.from_numpy(sT), s0

    def backward(self, x, ctx, dy, dsT):
        import oracle
        g = oracle.backward(*(x[n] for n in "rwkvab"), dy, s0=ctx, dsT=dsT)
        return {k: torch.from_numpy(v) for k, v in g.items()}

    def state_grad(self, x, ctx, dy):
        return self.backward(x, ctx, dy, None)["ds0"]

    def scan(self, M, C, init, backward):
        B, nseg, H = M.shape[:3]
        S = torch.zeros((B, H, N, N), dtype=M.dtype) if init is None else init.to(M.dtype).clone()
        out = torch.empty_like(M)
        order = range(nseg - 1, -1, -1) if backward else range(nseg)
        for k in order:
            out[:, k] = S
            S = C[:, k] + (S @ M[:, k].transpose(-1, -2) if backward else S @ M[:, k])
        return out, S


def _worker(rank, world, port, use_gpu, nseg, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import oracle
    from rwkv_linear_attention_wkv7_gb300 import seqpar, synthetic
    from tests import parity
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = synthetic.WorkloadSpec("seqpar", 2, 64 * world, 2, dtype="bf16" if use_gpu else "f32", s0_std=0.1,
                                      with_dsT=True, seed=11)
        full = synthetic.make_inputs(spec)
        tr = spec.T // world
        sl = slice(rank * tr, (rank + 1) * tr)
        dev = "cuda:0" if use_gpu else "cpu"
        x = {n: full[n][:, sl].contiguous().to(dev) for n in "rwkvab"}
        dy = full["dy"][:, sl].contiguous().to(dev)
        s0, dsT = full["s0"].to(dev), full["dsT"].to(dev)
        if use_gpu:
            from rwkv_linear_attention_wkv7_gb300 import build
            build()
            torch.cuda.set_device(0)
            solver = seqpar.CudaSpanSolver(nseg=nseg)
        else:
            solver = OracleSpanSolver()
        y, sT, ctx = seqpar.forward(x, s0=s0, solver=solver)
        g = seqpar.backward(x, ctx, dy, dsT=dsT, solver=solver)
        if use_gpu:
            torch.cuda.synchronize()
        ry, rsT, _ = oracle.forward(*(full[n] for n in "rwkvab"), s0=full["s0"], L=16, want_ckpt=False)
        rg = oracle.backward(*(full[n] for n in "rwkvab"), full["dy"], s0=full["s0"], dsT=full["dsT"])
        errs = {"y": parity.max_rel(y.double().cpu().numpy(), ry[:, sl]),
                "sT": parity.max_rel(sT.double().cpu().numpy(), rsT),
                "ds0": parity.grad_rel(g["ds0"].double().cpu().numpy(), rg["ds0"])}
        for n in parity.GRADS:
            errs[n] = parity.grad_rel(g[n].double().cpu().numpy(), rg[n][:, sl])
        out[rank] = errs
    finally:
        dist.destroy_process_group()


def _run(use_gpu, world=2, nseg=2):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, use_gpu, nseg, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    return dict(out)


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_oracle_spans(world):
    """The exchange with the oracle as the span solver reproduces the
    whole-sequence oracle to float64 rounding (every rank's span, sT, ds0)."""
    res = _run(use_gpu=False, world=world)
    assert sorted(res) == list(range(world))
    for rank, errs in res.items():
        for k, e in errs.items():
            assert e < 1e-11, (rank, k, e)


@pytest.mark.gpu
@pytest.mark.parametrize("nseg", [1, 2])
def test_world2_on_one_gpu(nseg):
    """Both ranks on cuda:0 with the library's kernels (two spans of 64 tokens;
    nseg 1: the summaries from the state passes, nseg 2: each span cut into 2
    segments), against the whole-sequence oracle at the parity bars."""
    from tests import parity
    res = _run(use_gpu=True, nseg=nseg)
    for rank, errs in res.items():
        assert errs["y"] <= parity.FWD_TOL and errs["sT"] <= parity.FWD_TOL, (rank, errs)
        for k in parity.GRADS + ("ds0",):
            assert errs[k] <= parity.GRAD_TOL, (rank, k, errs[k])
