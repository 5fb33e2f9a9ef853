#!/usr/bin/env python3
"""WKV7 forward+backward throughput on GB300.

One step = wkv7_forward (y, sT, checkpoints every L=16 tokens) + wkv7_backward
(all six input gradients and ds0) over one batch of the workload
B=16, T=4096, H=32, N=64 with bf16 r/w/k/v/a/b and fp32 state, outputs and
gradients (synthetic seeded inputs).  Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica of the batch (heads are
independent; no data-path collective): weak scaling, value = all ranks'
tokens / max-over-ranks time.  ``--impl reference`` times the fp64 CPU
oracle on this host's cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from rwkv_linear_attention_wkv7_gb300 import synthetic  # noqa: E402

METRIC = "WKV7 fwd+bwd tokens/sec at B=16,T=4096,H=32,N=64; % HBM roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "bf16_b16_t4096_h32"
DECODE_WORKLOAD = "decode_b512_h32"
TIMESPLIT_WORKLOAD = "long_b1_t65536_h8"
TIMESPLIT_SEGMENTS = 64
INPUTS = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")
L2_BYTES = 126 * 2**20


def esize(spec):
    return 2 if spec.dtype == "bf16" else 4


def algorithmic_bytes(spec):
    """Bytes a launch must move at minimum (checkpoints excluded: they are an
    implementation choice).  Forward: 6 inputs + y (+ s0, sT).  Backward:
    6 inputs + dy + 6 gradients (+ dsT, ds0)."""
    E = spec.elems
    st = spec.B * spec.H * spec.N * spec.N * 4
    fwd = E * (6 * esize(spec) + 4) + st * (2 if spec.s0_std > 0 else 1)
    bwd = E * (6 * esize(spec) + 4 + 6 * 4) + st * (2 if spec.with_dsT else 1)
    return fwd, bwd


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_traffic(workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on this workload and on the chunked kernels as they are now (the hash of
    their source files is recorded with it)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return {}
    try:
        with open(p) as f:
            d = json.loads("".join(l for l in f if not l.startswith("#")))
    except ValueError:
        return {}
    from rwkv_linear_attention_wkv7_gb300 import _build
    if d.get("workload") != workload or d.get("source_hash") != _build.source_hash(_build.CHUNK_KERNEL_FILES):
        return {}
    return d.get("kernels", {})


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.TemporaryFile(mode="w+")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle leg

def oracle_sample(spec, host_heads, n_heads, threads):
    """Time the fp64 oracle (fwd+bwd over all T) on n_heads heads; returns
    (seconds, tokens) where tokens = head-tokens / H."""
    import oracle
    heads = list(host_heads.keys())[:n_heads]

    def one(b, h):
        x = host_heads[(b, h)]
        oracle.forward(*(x[n] for n in INPUTS), s0=x.get("s0"), L=spec.L)
        oracle.backward(*(x[n] for n in INPUTS), x["dy"], s0=x.get("s0"), dsT=x.get("dsT"))

    t0 = time.perf_counter()
    oracle.per_head(one, heads, threads)
    dt = time.perf_counter() - t0
    return dt, len(heads) * spec.T / spec.H


def host_head_slices(spec, n):
    """Draw the workload's inputs and keep n heads' slices on the host as float64-ready tensors."""
    import numpy as np
    g = np.random.default_rng(1)
    picks = []
    while len(picks) < min(n, spec.B * spec.H):
        bh = (int(g.integers(0, spec.B)), int(g.integers(0, spec.H)))
        if bh not in picks:
            picks.append(bh)
    out = {bh: {} for bh in picks}
    for name, t in synthetic.stream_inputs(spec):
        for bh in picks:
            out[bh][name] = synthetic.head_slice(t, *bh, state=name in ("s0", "dsT"))
    return out


def cpu_baseline(spec, target_s=12.0, host_heads=None):
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    if host_heads is None:
        host_heads = host_head_slices(spec, min(spec.B * spec.H, max(cores * 8, 16)))
    t1, _ = oracle_sample(spec, host_heads, 1, 1)  # calibrate one head on one core
    n = max(1, min(len(host_heads), int(target_s * cores / max(t1, 1e-3))))
    dt, toks = oracle_sample(spec, host_heads, n, cores)
    return {"value": toks / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of {spec.B * spec.H} (b,h) heads, full T={spec.T}, fwd+bwd in fp64; "
                      f"tokens counted as head-tokens/H; {dt:.1f} s wall"}, dt


def run_reference(args, world, rank):
    spec = workload_of(args)
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    host_heads = host_head_slices(spec, cores)
    n = min(len(host_heads), cores)
    for _ in range(args.warmup):
        oracle_sample(spec, host_heads, 1, 1)
    times, toks = [], 0.0
    for _ in range(args.steps):
        dt, tk = oracle_sample(spec, host_heads, n, cores)
        times.append(dt)
        toks = tk
    value = toks * len(times) / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(spec, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: {n} (b,h) heads of {spec.B * spec.H}, full T={spec.T}, "
                                       "fwd+bwd fp64 oracle on all host cores"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(spec, args):
    return {"workload": spec.name, "B": spec.B, "T": spec.T, "H": spec.H, "N": spec.N,
            "input_dtype": spec.dtype, "state_dtype": "f32", "ckpt_stride": spec.L,
            "factor_cache": spec.L == 16,
            "parallelism": f"replicas x{args.gpus} (independent heads)",
            "l2": f"inputs larger than L2 ({spec.elems * 6 * esize(spec) / 1e9:.2f} GB of r..b per step), no flush"}


# ------------------------------------------------------------------ GPU leg

def workload_of(args):
    spec = synthetic.WORKLOADS[args.workload]
    import dataclasses
    if args.batch:
        spec = dataclasses.replace(spec, B=args.batch, name=f"{spec.name}@B={args.batch}")
    if args.seq_len:
        spec = dataclasses.replace(spec, T=args.seq_len, name=f"{spec.name}@T={args.seq_len}")
    return spec


def bench_decode(wkv7, dev, stream, peak, world, steps=200, warmup=5):
    """Batched streaming decode: B sequences advance one token per call from a
    carried state of B*H heads, updated in place.  The state (B*H*16 KiB) is
    larger than L2, so every call reads and writes it in HBM; the token
    vectors cycle over the workload's T drawn sets."""
    spec = synthetic.DECODE_WORKLOADS[DECODE_WORKLOAD]
    d = synthetic.make_inputs(spec, device=dev)
    toks = [[d[n][:, t].contiguous() for n in INPUTS] for t in range(spec.T)]
    state = d["s0"]
    del d
    y = torch.empty((spec.B, spec.H, spec.N), device=dev)

    def go(i):
        wkv7.decode_step(*toks[i % spec.T], state, y=y, stream=stream)

    for i in range(warmup):
        go(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        go(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world) / steps
    es = 2 if spec.dtype == "bf16" else 4
    heads = spec.B * spec.H
    per_step = heads * (2 * spec.N * spec.N * 4 + 6 * spec.N * es + spec.N * 4)  # state in + out, vectors, y
    gbs = per_step / (ms / 1e3) / 1e9
    return {"workload": spec.name, "B": spec.B, "H": spec.H, "N": spec.N, "input_dtype": spec.dtype,
            "tokens_per_s": world * spec.B / (ms / 1e3), "us_per_step": ms * 1e3, "steps": steps,
            "launches": steps,
            "roofline": {"bound": "hbm", "kernel": "wkv7 decode", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "algorithmic_bytes": per_step},
            "l2": f"state ({heads * spec.N * spec.N * 4 / 1e6:.0f} MB) larger than L2, no flush"}


def bench_timesplit(wkv7, dev, stream, peak, world, steps=3, warmup=1):
    """Few, long sequences (8 heads of 65536 tokens): the plain entry points
    (one thread block per head) against the time-split ones (each sequence in
    TIMESPLIT_SEGMENTS segments side by side), fwd+bwd per step, with the
    largest relative difference between the two results."""
    spec = synthetic.TIMESPLIT_WORKLOADS[TIMESPLIT_WORKLOAD]
    d = synthetic.make_inputs(spec, device=dev)
    xs = [d[n] for n in INPUTS]
    B, T, H, N = spec.B, spec.T, spec.H, spec.N
    nseg = TIMESPLIT_SEGMENTS
    outs = {"y": torch.empty((B, T, H, N), device=dev), "sT": torch.empty((B, H, N, N), device=dev),
            "ckpt": torch.empty((B, H, wkv7.ckpt_count(T, 16), N, N), device=dev),
            "factors": torch.empty((B, H, wkv7.factor_floats(T)), device=dev)}
    g_plain = {n: torch.empty((B, T, H, N), device=dev) for n in GRADS}
    g_plain["ds0"] = torch.empty((B, H, N, N), device=dev)
    ws = torch.empty(wkv7.timesplit_workspace_floats(B, T, H, nseg), device=dev)
    so = {"y": torch.empty((B, T, H, N), device=dev), "sT": torch.empty((B, H, N, N), device=dev)}
    g_split = {n: torch.empty_like(v) for n, v in g_plain.items()}

    def plain():
        wkv7.forward(*xs, s0=d["s0"], L=16, want_factors=True, out=outs, stream=stream)
        wkv7.backward(*xs, outs["ckpt"], d["dy"], dsT=d["dsT"], L=16, factors=outs["factors"], out=g_plain,
                      stream=stream)

    def split():
        wkv7.forward_timesplit(*xs, s0=d["s0"], nseg=nseg, workspace=ws, out=so, stream=stream)
        wkv7.backward_timesplit(*xs, d["dy"], dsT=d["dsT"], nseg=nseg, workspace=ws, out=g_split, stream=stream)

    res = {}
    for name, fn in (("plain", plain), ("split", split)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = max_over_ranks(e0.elapsed_time(e1), world) / steps
    wkv7.async_status()

    def rel(a, b):
        return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))
    diff = max([rel(so["y"], outs["y"]), rel(so["sT"], outs["sT"])] + [rel(g_split[n], g_plain[n]) for n in g_plain])
    fwd_b, bwd_b = algorithmic_bytes(spec)
    gbs = (fwd_b + bwd_b) / (res["split"] / 1e3) / 1e9
    return {"workload": spec.name, "B": B, "T": T, "H": H, "input_dtype": spec.dtype, "segments": nseg,
            "plain_ms_per_step": res["plain"], "split_ms_per_step": res["split"],
            "plain_tokens_per_s": world * spec.tokens / (res["plain"] / 1e3),
            "split_tokens_per_s": world * spec.tokens / (res["split"] / 1e3),
            "split_hbm_fraction_step": gbs / peak, "max_rel_diff_split_vs_plain": diff, "steps": steps}


def run_ours(args, world, rank, local):
    from rwkv_linear_attention_wkv7_gb300 import build, wkv7
    build()
    spec = workload_of(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    # inputs: drawn on the host (seeded), moved to HBM before timing
    host_heads = {}
    want_cpu = rank == 0 and not args.no_cpu
    cores = os.cpu_count() or 1
    n_keep = min(spec.B * spec.H, max(cores * 32, 16)) if want_cpu else 0
    import numpy as np
    g = np.random.default_rng(1)
    keep = []
    while len(keep) < n_keep:
        bh = (int(g.integers(0, spec.B)), int(g.integers(0, spec.H)))
        if bh not in keep:
            keep.append(bh)
    host_heads = {bh: {} for bh in keep}
    d = {}
    pinned = {}
    for name, t in synthetic.stream_inputs(spec):
        for bh in keep:
            host_heads[bh][name] = None if t is None else synthetic.head_slice(t, *bh, state=name in ("s0", "dsT"))
        d[name] = None if t is None else t.to(dev)
        if not args.no_e2e and t is not None and name in INPUTS + ("dy",):
            pinned[name] = t.pin_memory()
        del t

    B, T, H, N = spec.B, spec.T, spec.H, spec.N
    nck = wkv7.ckpt_count(T, spec.L)
    use_fac = spec.L == 16
    outs = {"y": torch.empty((B, T, H, N), device=dev), "sT": torch.empty((B, H, N, N), device=dev),
            "ckpt": torch.empty((B, H, nck, N, N), device=dev)}
    if use_fac:  # the forward's per-chunk factor cache, reused by the backward
        outs["factors"] = torch.empty((B, H, wkv7.factor_floats(T)), device=dev)
    gouts = {n: torch.empty((B, T, H, N), device=dev) for n in GRADS}
    gouts["ds0"] = torch.empty((B, H, N, N), device=dev)
    stream = torch.cuda.current_stream(dev)

    ev_f = []  # per-launch events (forward, backward) on the launching stream

    def step(record=False):
        if record:
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
        wkv7.forward(*(d[n] for n in INPUTS), s0=d["s0"], L=spec.L, want_factors=use_fac, out=outs, stream=stream)
        if record:
            e1.record(stream)
        wkv7.backward(*(d[n] for n in INPUTS), outs["ckpt"], d["dy"], dsT=d["dsT"], L=spec.L,
                      factors=outs.get("factors"), out=gouts, stream=stream)
        if record:
            e2.record(stream)
            ev_f.append((e0, e1, e2))

    # The step as a user runs it: wkv7_forward_backward, the forward and the
    # backward as concurrent blocks of batch rows (the library's default split)
    # on its own streams, forked from and joined back into this stream.  The
    # workloads with another checkpoint stride run the two calls in a row.
    use_step = spec.L == 16
    fbout = {**outs, **gouts}
    nsplit = args.nsplit  # 0: the library's default
    split = wkv7.forward_backward_blocks(B, spec.T, spec.H, nsplit) if use_step else 1
    launches_per_step = 2 * split

    def fb_step():
        if use_step:
            wkv7.forward_backward(*(d[n] for n in INPUTS), d["dy"], s0=d["s0"], dsT=d["dsT"], want_factors=use_fac,
                                  nsplit=nsplit, out=fbout, stream=stream)
        else:
            step()

    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(args.warmup):
        fb_step()
    w1.record(stream)
    torch.cuda.synchronize()
    # the timed region repeats whole rounds of K steps until it lasts at least
    # --min-timed-s, so that the clock record sampled during it has several samples
    # (every round is K full steps; ms_per_step divides by all timed steps)
    warm_ms = max_over_ranks(w0.elapsed_time(w1) / max(args.warmup, 1), world)
    # (a 15 % margin: warm-up steps can run a little slower than timed ones)
    rounds = max(1, -(-int(1.15 * args.min_timed_s * 1e3) // max(int(warm_ms * args.steps), 1)))
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(rounds * args.steps):
            fb_step()
        t_end.record(stream)
        torch.cuda.synchronize()
    wkv7.async_status()  # raises if a kernel's bounded wait on its bulk copies ran out
    barrier(world)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    clocks = clk.summary()

    # each kernel on its own: the same step as wkv7_forward then wkv7_backward on
    # the whole batch, CUDA events around every launch (the roofline's launch times)
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    s0_ev, s1_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0_ev.record(stream)
    for _ in range(args.steps):
        step(record=True)
    s1_ev.record(stream)
    torch.cuda.synchronize()
    wkv7.async_status()
    seq_step_ms = max_over_ranks(s0_ev.elapsed_time(s1_ev), world) / args.steps
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in ev_f)
    bwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in ev_f)

    ms_step = total_ms / (rounds * args.steps)

    # head to head: the same backward launches with two of the 64-row state
    # products on the tensor cores (tcgen05) instead of warp-level mma.sync
    bwd_tc_ms = None
    if spec.L == 16:
        os.environ["WKV7_BACKWARD_KERNEL"] = "tcgen05"
        try:
            def bwd_only():
                wkv7.backward(*(d[n] for n in INPUTS), outs["ckpt"], d["dy"], dsT=d["dsT"], L=spec.L,
                              factors=outs.get("factors"), out=gouts, stream=stream)
            for _ in range(2):
                bwd_only()
            m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            m0.record(stream)
            for _ in range(args.steps):
                bwd_only()
            m1.record(stream)
            torch.cuda.synchronize()
            bwd_tc_ms = max_over_ranks(m0.elapsed_time(m1), world) / args.steps
        finally:
            del os.environ["WKV7_BACKWARD_KERNEL"]
        wkv7.async_status()
    value = world * spec.tokens / (ms_step / 1e3)
    peak, peak_kind = load_peaks()
    fwd_bytes, bwd_bytes = algorithmic_bytes(spec)
    traffic = load_traffic(spec.name)
    dom = "backward" if bwd_ms >= fwd_ms else "forward"
    dom_ms, dom_bytes = (bwd_ms, bwd_bytes) if dom == "backward" else (fwd_ms, fwd_bytes)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    step_gbs = (fwd_bytes + bwd_bytes) / (ms_step / 1e3) / 1e9

    # end to end through the public API with host buffers: every step copies
    # its inputs and dy from pinned host memory, runs forward + backward, and
    # copies y and the six gradients back.  Steps are pipelined over three
    # streams (H2D | compute | D2H) with two device buffer sets, so step k's
    # copies overlap step k-1's compute and each other (the host link is
    # full duplex); the sequential form is reported beside it.
    e2e = None
    if not args.no_e2e:
        host_out = {n: torch.empty(outs["y"].shape, pin_memory=True) for n in ("y",) + GRADS}
        h2d = sum(pinned[n].numel() * pinned[n].element_size() for n in pinned)
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())

        # The step through wkv7_forward_backward with one block (its two calls in order on
        # this stream): the copies bound this pipeline, so the split gains nothing here,
        # and a stream of the library's beside the two copy streams made the overlap
        # come and go from run to run (22 to 37 ms per step).
        def run_step(din, o, gq):
            if use_step:
                wkv7.forward_backward(*(din.get(n, d[n]) for n in INPUTS), din["dy"], s0=d["s0"], dsT=d["dsT"],
                                      want_factors=use_fac, nsplit=1, out={**o, **gq}, stream=stream)
                return
            wkv7.forward(*(din.get(n, d[n]) for n in INPUTS), s0=d["s0"], L=spec.L, want_factors=use_fac, out=o,
                         stream=stream)
            wkv7.backward(*(din.get(n, d[n]) for n in INPUTS), o["ckpt"], din["dy"], dsT=d["dsT"], L=spec.L,
                          factors=o.get("factors"), out=gq, stream=stream)

        sets = []
        for k in range(2):
            din = {n: (d[n] if k == 0 else torch.empty_like(d[n])) for n in pinned}
            o = dict(outs)
            gq = dict(gouts)
            if k:
                o["y"] = torch.empty_like(outs["y"])
                for n in GRADS:
                    gq[n] = torch.empty_like(gouts[n])
            sets.append((din, o, gq))
        sh, sd = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        h_ev = [torch.cuda.Event() for _ in range(2)]
        c_ev = [torch.cuda.Event() for _ in range(2)]
        d_ev = [torch.cuda.Event() for _ in range(2)]

        def e2e_pipe(k):
            s = k % 2
            din, o, gq = sets[s]
            with torch.cuda.stream(sh):
                if k >= 2:
                    sh.wait_event(c_ev[s])  # step k-2 has read this input set
                for n in pinned:
                    din[n].copy_(pinned[n], non_blocking=True)
                h_ev[s].record(sh)
            stream.wait_event(h_ev[s])
            if k >= 2:
                stream.wait_event(d_ev[s])  # step k-2's results have left this output set
            run_step(din, o, gq)
            c_ev[s].record(stream)
            with torch.cuda.stream(sd):
                sd.wait_event(c_ev[s])
                host_out["y"].copy_(o["y"], non_blocking=True)
                for n in GRADS:
                    host_out[n].copy_(gq[n], non_blocking=True)
                d_ev[s].record(sd)

        def e2e_seq():
            din, o, gq = sets[0]
            for n in pinned:
                din[n].copy_(pinned[n], non_blocking=True)
            run_step(din, o, gq)
            host_out["y"].copy_(o["y"], non_blocking=True)
            for n in GRADS:
                host_out[n].copy_(gq[n], non_blocking=True)

        for k in range(2):
            e2e_pipe(k)
        e2e_seq()
        torch.cuda.synchronize()
        barrier(world)
        n_e2e = 24  # steady state: the first inputs in and the last results out are paid once
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(sh)
        for k in range(n_e2e):
            e2e_pipe(k)
        stream.wait_event(d_ev[(n_e2e - 1) % 2])
        a1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a0.elapsed_time(a1), world) / n_e2e
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(3):
            e2e_seq()
        b1.record(stream)
        torch.cuda.synchronize()
        seq_ms = max_over_ranks(b0.elapsed_time(b1), world) / 3
        wkv7.async_status()
        # the host link itself: one output tensor out, and dy in, each alone and both at
        # once; the step's copies cannot take less than link_bound_ms
        yb = host_out["y"].numel() * 4
        dyb = pinned["dy"].numel() * pinned["dy"].element_size()
        dsts = sets[0][0]["dy"]

        def timed(fn):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            fn()
            torch.cuda.synchronize()
            e[0].record(stream)
            fn()
            e[1].record(stream)
            torch.cuda.synchronize()
            return e[0].elapsed_time(e[1]) / 1e3

        def both():
            with torch.cuda.stream(sd):
                sd.wait_stream(stream)
                host_out["y"].copy_(outs["y"], non_blocking=True)
            dsts.copy_(pinned["dy"], non_blocking=True)
            stream.wait_stream(sd)

        d2h_gbs = yb / timed(lambda: host_out["y"].copy_(outs["y"], non_blocking=True)) / 1e9
        h2d_gbs = dyb / timed(lambda: dsts.copy_(pinned["dy"], non_blocking=True)) / 1e9
        both_gbs = (yb + dyb) / timed(both) / 1e9
        # neither direction beats its own rate, nor both together their joint rate
        link_ms = 1e3 * max(d2h / (d2h_gbs * 1e9), h2d / (h2d_gbs * 1e9), (h2d + d2h) / (both_gbs * 1e9))
        e2e = {"value": world * spec.tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": n_e2e, "pipelined": True,
               "sequential_ms_per_step": seq_ms, "entry": "wkv7_forward_backward, one block" if use_step else
               "wkv7_forward + wkv7_backward",
               "link": {"d2h_gbs": d2h_gbs, "h2d_gbs": h2d_gbs, "both_directions_gbs": both_gbs,
                        "link_bound_ms": link_ms, "frac_of_link_bound": link_ms / e2e_ms}}

    # the producers fused into the entry points: the same step through
    # wkv7_forward_fused / wkv7_backward_fused on the same draws taken before the
    # producers (w_pre, kk, avec in place of w, a, b; same bytes per element)
    fused = None
    if not args.no_fused and use_fac:
        fz = {}
        for name, t in synthetic.stream_inputs(spec, fused=True):
            if name in ("w_pre", "kk", "avec"):
                fz[name] = t.to(dev)
            del t
        fx = [d["r"], fz["w_pre"], d["k"], d["v"], fz["kk"], fz["avec"]]
        fg = {fn: gouts[gn] for fn, gn in zip(wkv7.FUSED_GRAD_NAMES, GRADS)}
        fg["ds0"] = gouts["ds0"]
        fev = []

        def fstep(record=False):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if record else None
            if record:
                e[0].record(stream)
            wkv7.forward_fused(*fx, s0=d["s0"], L=spec.L, want_factors=True, out=outs, stream=stream)
            if record:
                e[1].record(stream)
            wkv7.backward_fused(*fx, outs["ckpt"], d["dy"], dsT=d["dsT"], L=spec.L, factors=outs["factors"],
                                out=fg, stream=stream)
            if record:
                e[2].record(stream)
                fev.append(e)

        for _ in range(args.warmup):
            fstep()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            fstep(record=True)
        f1.record(stream)
        torch.cuda.synchronize()
        wkv7.async_status()
        f_ms = max_over_ranks(f0.elapsed_time(f1), world) / args.steps
        ff = statistics.mean(a.elapsed_time(b) for a, b, _ in fev)
        fb = statistics.mean(b.elapsed_time(c) for _, b, c in fev)
        # the same step in one call, the library's blocks of batch rows (wkv7_forward_backward_fused)
        fbo = {**outs, **fg}
        fblocks = wkv7.forward_backward_blocks(B, spec.T, spec.H, 0)

        def fcall():
            wkv7.forward_backward_fused(*fx, d["dy"], s0=d["s0"], dsT=d["dsT"], nsplit=0, out=fbo, stream=stream)

        for _ in range(args.warmup):
            fcall()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(args.steps):
            fcall()
        c1.record(stream)
        torch.cuda.synchronize()
        wkv7.async_status()
        fc_ms = max_over_ranks(c0.elapsed_time(c1), world) / args.steps
        # the same step with the producers and epilogues as separate elementwise
        # passes around the plain entry points (torch ops writing w, a, b to HBM
        # and reading the plain gradients back), for comparison
        dt_in = d["r"].dtype

        def ustep():
            sig = torch.sigmoid(fz["w_pre"].float())
            w = torch.exp(-synthetic.DECAY_COEFF * sig)
            kk32 = fz["kk"].float()
            a, b = (-kk32).to(dt_in), (kk32 * fz["avec"].float()).to(dt_in)
            wkv7.forward(d["r"], w.to(dt_in), d["k"], d["v"], a, b, s0=d["s0"], L=spec.L, want_factors=True,
                         out=outs, stream=stream)
            gg = wkv7.backward(d["r"], w.to(dt_in), d["k"], d["v"], a, b, outs["ckpt"], d["dy"], dsT=d["dsT"],
                               L=spec.L, factors=outs["factors"], out=gouts, stream=stream)
            gw = gg["dw"] * w * (-synthetic.DECAY_COEFF) * sig * (1.0 - sig)
            gk = -gg["da"] + fz["avec"].float() * gg["db"]
            ga = kk32 * gg["db"]
            return gw, gk, ga

        for _ in range(args.warmup):
            ustep()
        torch.cuda.synchronize()
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_u = max(3, args.steps // 10)
        u0.record(stream)
        for _ in range(n_u):
            ustep()
        u1.record(stream)
        torch.cuda.synchronize()
        u_ms = max_over_ranks(u0.elapsed_time(u1), world) / n_u
        fused = {"ms_per_step": fc_ms, "tokens_per_s": world * spec.tokens / (fc_ms / 1e3),
                 "entry": f"wkv7_forward_backward_fused, {fblocks} blocks of batch rows", "launches_per_step": 2 * fblocks,
                 "sequential_ms_per_step": f_ms, "forward_ms": ff, "backward_ms": fb,
                 "separate_producers_ms_per_step": u_ms,
                 "roofline": {"bound": "hbm", "kernel": "wkv7 backward (fused producers)",
                              "achieved": bwd_bytes / (fb / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                              "frac": bwd_bytes / (fb / 1e3) / 1e9 / peak, "algorithmic_bytes": bwd_bytes},
                 "inputs": "r, w_pre, k, v, kk, avec (w, a, b computed in the kernels)"}
        del fz, fx

    # the GroupNorm + bonus output epilogue fused into the step (wkv7_forward_gn +
    # wkv7_backward_gn, do = the same dy draw), beside the plain step with the
    # epilogue as separate torch passes (group_norm and the bonus, and their
    # autograd backward) around the plain entry points
    gnres = None
    if not args.no_gn and use_fac:
        gp = {n: t.to(dev) for n, t in synthetic.gn_params(H, seed=0).items()}
        xs = [d[n] for n in INPUTS]
        go = {"y": outs["y"], "o": torch.empty_like(outs["y"]), "sT": outs["sT"], "ckpt": outs["ckpt"],
              "factors": outs["factors"]}
        gg = dict(gouts)
        gg.update({n: torch.empty((H, N), device=dev) for n in ("dgn_w", "dgn_b", "dr_k")})
        gws = torch.empty(wkv7.gn_workspace_floats(B, H), device=dev)
        gev = []

        def gstep(record=False):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if record else None
            if record:
                e[0].record(stream)
            wkv7.forward_gn(*xs, gp["gn_w"], gp["gn_b"], gp["r_k"], s0=d["s0"], L=16, out=go, stream=stream)
            if record:
                e[1].record(stream)
            wkv7.backward_gn(*xs, go["ckpt"], go["factors"], go["y"], d["dy"], gp["gn_w"], gp["r_k"], dsT=d["dsT"],
                             workspace=gws, out=gg, stream=stream)
            if record:
                e[2].record(stream)
                gev.append(e)

        for _ in range(args.warmup):
            gstep()
        torch.cuda.synchronize()
        barrier(world)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            gstep(record=True)
        g1.record(stream)
        torch.cuda.synchronize()
        wkv7.async_status()
        g_ms = max_over_ranks(g0.elapsed_time(g1), world) / args.steps
        gf = statistics.mean(a.elapsed_time(b) for a, b, _ in gev)
        gb = statistics.mean(b.elapsed_time(c) for _, b, c in gev)
        # the same step in one call, the library's blocks of batch rows (wkv7_forward_backward_gn)
        gbo = {**go, **gg}
        gblocks = wkv7.forward_backward_blocks(B, spec.T, spec.H, 0)

        def gcall():
            wkv7.forward_backward_gn(*xs, d["dy"], gp["gn_w"], gp["gn_b"], gp["r_k"], s0=d["s0"], dsT=d["dsT"],
                                     nsplit=0, workspace=gws, out=gbo, stream=stream)

        for _ in range(args.warmup):
            gcall()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(args.steps):
            gcall()
        c1.record(stream)
        torch.cuda.synchronize()
        wkv7.async_status()
        gc_ms = max_over_ranks(c0.elapsed_time(c1), world) / args.steps

        def sstep():
            y_, _, ck_, fac_ = wkv7.forward(*xs, s0=d["s0"], L=16, want_factors=True, out=outs, stream=stream)
            yv = y_.detach().requires_grad_(True)
            o_ = torch.nn.functional.group_norm(yv.reshape(B * T, H * N), H, gp["gn_w"].reshape(-1),
                                                gp["gn_b"].reshape(-1), eps=64e-5).reshape(B, T, H, N)
            o_ = o_ + (xs[0].float() * xs[2].float() * gp["r_k"]).sum(-1, keepdim=True) * xs[3].float()
            o_.backward(d["dy"])
            wkv7.backward(*xs, ck_, yv.grad, dsT=d["dsT"], L=16, factors=fac_, out=gouts, stream=stream)

        for _ in range(2):
            sstep()
        torch.cuda.synchronize()
        s0_, s1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_s = max(3, args.steps // 10)
        s0_.record(stream)
        for _ in range(n_s):
            sstep()
        s1_.record(stream)
        torch.cuda.synchronize()
        sep_ms = max_over_ranks(s0_.elapsed_time(s1_), world) / n_s
        gbytes = bwd_bytes + spec.elems * 4  # + the forward's y, read back by the epilogue's backward
        gnres = {"ms_per_step": gc_ms, "tokens_per_s": world * spec.tokens / (gc_ms / 1e3),
                 "entry": f"wkv7_forward_backward_gn, {gblocks} blocks of batch rows",
                 "launches_per_step": 2 * gblocks + 1, "sequential_ms_per_step": g_ms, "forward_ms": gf,
                 "backward_ms": gb, "separate_epilogue_ms_per_step": sep_ms,
                 "roofline": {"bound": "hbm", "kernel": "wkv7 backward with the epilogue's backward",
                              "achieved": gbytes / (gb / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                              "frac": gbytes / (gb / 1e3) / 1e9 / peak, "algorithmic_bytes": gbytes},
                 "outputs": "o (GroupNorm + bonus) and y; dgn_w, dgn_b, dr_k beside the seven gradients"}
        del go, gg, gws

    timesplit = None
    if not args.no_timesplit:
        timesplit = bench_timesplit(wkv7, dev, stream, peak, world)

    decode = None
    if not args.no_decode:
        decode = bench_decode(wkv7, dev, stream, peak, world)
        wkv7.async_status()

    cpu = None
    if want_cpu:
        cpu, _ = cpu_baseline(spec, host_heads=host_heads)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "rounds": rounds, "timed_steps": rounds * args.steps, "timed_ms": total_ms,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config_of(spec, args),
        "roofline": {"bound": "hbm", "kernel": f"wkv7 {dom}", "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic.get(dom), "algorithmic_bytes": dom_bytes, "launch_ms": dom_ms},
        "hbm_fraction_step": step_gbs / peak,
        "step": {"entry": "wkv7_forward_backward" if use_step else "wkv7_forward + wkv7_backward",
                 "blocks_of_batch_rows": split, "launches": launches_per_step,
                 "sequential_ms_per_step": seq_step_ms,
                 "sequential": "wkv7_forward then wkv7_backward on the whole batch, one stream"},
        "forward": {"ms": fwd_ms, "tokens_per_s": spec.tokens / (fwd_ms / 1e3),
                    "algorithmic_gbs": fwd_bytes / (fwd_ms / 1e3) / 1e9},
        "backward": {"ms": bwd_ms, "algorithmic_gbs": bwd_bytes / (bwd_ms / 1e3) / 1e9,
                     "kernel": "mma.sync", "tcgen05_variant_ms": bwd_tc_ms},
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches_per_step * rounds * args.steps, "clocks": clocks,
        "fused": fused, "gn_epilogue": gnres, "decode": decode, "timesplit": timesplit,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None,
                    help="override B of the workload (smaller profiling cases of the same kernels)")
    ap.add_argument("--seq-len", type=int, default=None, help="override T of the workload (profiling cases)")
    ap.add_argument("--nsplit", type=int, default=0, choices=range(5),
                    help="blocks of batch rows of the one-call step (0: the library's default)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the batched decode measurement")
    ap.add_argument("--no-fused", action="store_true", help="skip the fused-producer measurement")
    ap.add_argument("--no-timesplit", action="store_true", help="skip the time-split measurement")
    ap.add_argument("--no-gn", action="store_true", help="skip the fused output-epilogue measurement")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="repeat rounds of --steps steps until the timed region lasts this long (0: one round)")
    args = ap.parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
