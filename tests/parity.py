"""Helpers for GPU-vs-oracle parity: run both sides on the same seeded inputs
and compare with the tolerances the library promises.

Forward (y, sT, checkpoints): max |gpu - ref| <= 2e-4 * max |ref| per tensor
and per (b,h).  Gradients, per tensor and per (b,h), two bars that must both
hold: element by element, max |gpu - ref| <= 1e-3 * max |ref| (so that one bad
token or key column cannot hide in a norm), and ||gpu - ref||_F / ||ref||_F <=
1e-3 (the GPU-vs-CPU metric of the "cortiq_engine/fcd_ops.rs" page's
gemm_dx_gpu_matches_cpu test, with the bar relaxed from 1e-4 to 1e-3 because
the recurrence chains T dependent fp32 steps instead of one contraction).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from rwkv_linear_attention_wkv7_gb300 import synthetic, wkv7

FWD_TOL = 2e-4
GRAD_TOL = 1e-3
INPUTS = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")
# the fused entry points' inputs and gradients (producers computed inside)
INPUTS_FUSED = ("r", "w_pre", "k", "v", "kk", "avec")
GRADS_FUSED = ("dr", "dw_pre", "dk", "dv", "dkk", "davec")
STATE_KEYS = ("s0", "dsT", "sT", "ds0", "ckpt")


def to_dev(x, dev="cuda"):
    return None if x is None else x.to(dev).contiguous()


def inputs_on_device(spec, heads=None, dev="cuda", fused=False):
    """Draw ``spec``'s inputs, move each to the GPU as soon as it is drawn and
    keep on the host only the slices of ``heads`` (all heads if None)."""
    dev_in, host = {}, {}
    for name, t in synthetic.stream_inputs(spec, fused=fused):
        if t is None:
            dev_in[name] = None
            continue
        dev_in[name] = t.to(dev).contiguous()
        if heads is None:
            host[name] = t
        else:
            host[name] = {bh: synthetic.head_slice(t, *bh, state=name in STATE_KEYS) for bh in heads}
        del t
    return dev_in, host


def run_gpu(d, L=16, backward=True, factors=None, fused=False):
    """Forward (+ backward) through the C ABI on device inputs ``d``; outputs stay on the device.

    ``factors``: pass the forward's per-chunk factor cache to the backward
    (the training path); default: whenever L == 16, the stride it needs.
    ``fused``: the entry points with the producers fused in (inputs
    INPUTS_FUSED, gradients GRADS_FUSED)."""
    use_fac = (L == 16) if factors is None else factors
    if fused:
        res = wkv7.forward_fused(*(d[n] for n in INPUTS_FUSED), s0=d.get("s0"), L=L, want_factors=use_fac)
        out = {"y": res[0], "sT": res[1], "ckpt": res[2]}
        if backward:
            out.update(wkv7.backward_fused(*(d[n] for n in INPUTS_FUSED), res[2], d["dy"], dsT=d.get("dsT"), L=L,
                                           factors=res[3] if use_fac else None))
        torch.cuda.synchronize()
        wkv7.async_status()
        return out
    res = wkv7.forward(*(d[n] for n in INPUTS), s0=d.get("s0"), L=L, want_factors=use_fac)
    y, sT, ck = res[:3]
    fac = res[3] if use_fac else None
    out = {"y": y, "sT": sT, "ckpt": ck}
    if backward:
        out.update(wkv7.backward(*(d[n] for n in INPUTS), ck, d["dy"], dsT=d.get("dsT"), L=L, factors=fac))
    torch.cuda.synchronize()
    wkv7.async_status()  # no bounded wait on the kernels' bulk copies ran out
    return out


def _head_input(host, name, b, h):
    x = host.get(name)
    if x is None:
        return None
    if isinstance(x, dict):
        return x[(b, h)]
    return synthetic.head_slice(x, b, h, state=name in STATE_KEYS)


def oracle_head(host, b, h, L=16, backward=True, fused=False):
    """Oracle results for head (b, h) only, float64 numpy in B=H=1 shapes."""
    names = INPUTS_FUSED if fused else INPUTS
    fwd, bwd = (oracle.forward_fused, oracle.backward_fused) if fused else (oracle.forward, oracle.backward)
    sl = {n: _head_input(host, n, b, h) for n in names + ("s0", "dy", "dsT")}
    y, sT, ck = fwd(*(sl[n] for n in names), s0=sl["s0"], L=L)
    res = {"y": y, "sT": sT, "ckpt": ck}
    if backward:
        res.update(bwd(*(sl[n] for n in names), sl["dy"], s0=sl["s0"], dsT=sl["dsT"]))
    return res


def gpu_head(out, b, h):
    """Slice the GPU results to head (b, h) in the oracle's B=H=1 shapes (host float64)."""
    res = {}
    for k, v in out.items():
        if v is None:
            continue
        if k in STATE_KEYS:
            res[k] = v[b:b + 1, h:h + 1].double().cpu().numpy()
        else:
            res[k] = v[b:b + 1, :, h:h + 1].double().cpu().numpy()
    return res


def max_rel(got, ref):
    den = float(np.abs(ref).max()) if ref.size else 0.0
    num = float(np.abs(got - ref).max()) if ref.size else 0.0
    return num / den if den > 0 else num


def fro_rel(got, ref):
    den = float(np.linalg.norm(ref))
    num = float(np.linalg.norm(got - ref))
    return num / den if den > 0 else num


def grad_rel(got, ref):
    """The larger of the two gradient errors (element-wise max and rel-Frobenius)."""
    return max(max_rel(got, ref), fro_rel(got, ref))


def compare(gpu, ref, backward=True, what="", grads=GRADS):
    """Assert the tolerances; return the measured errors."""
    errs = {}
    for k in ("y", "sT", "ckpt"):
        if ref.get(k) is not None and k in gpu:
            errs[k] = max_rel(gpu[k], ref[k])
            assert errs[k] <= FWD_TOL, f"{what} {k}: max err {errs[k]:.3e} x max|ref| > {FWD_TOL}"
    if backward:
        for k in grads + ("ds0",):
            if k in gpu:
                fr, mx = fro_rel(gpu[k], ref[k]), max_rel(gpu[k], ref[k])
                errs[k] = max(fr, mx)
                assert mx <= GRAD_TOL, f"{what} {k}: max err {mx:.3e} x max|ref| > {GRAD_TOL} (rel Frobenius {fr:.3e})"
                assert fr <= GRAD_TOL, f"{what} {k}: rel Frobenius {fr:.3e} > {GRAD_TOL} (max err {mx:.3e})"
    return errs


def check_heads(host, out, heads, L=16, backward=True, threads=None, fused=False):
    """Oracle the given heads in parallel and compare each with the GPU result."""
    refs = oracle.per_head(lambda b, h: oracle_head(host, b, h, L=L, backward=backward, fused=fused), heads,
                           threads)
    worst = {}
    for (b, h), ref in zip(heads, refs):
        e = compare(gpu_head(out, b, h), ref, backward=backward, what=f"head (b={b}, h={h})",
                    grads=GRADS_FUSED if fused else GRADS)
        for k, v in e.items():
            worst[k] = max(worst.get(k, 0.0), v)
    return worst


def all_heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def sample_heads(B, H, n=6, seed=0):
    """Corners, the middle, and seeded random heads."""
    g = np.random.default_rng(seed)
    heads = {(0, 0), (B - 1, H - 1), (B // 2, H // 2)}
    while len(heads) < min(n, B * H):
        heads.add((int(g.integers(0, B)), int(g.integers(0, H))))
    return sorted(heads)


# ---- the GroupNorm + bonus output epilogue (wkv7_forward_gn / wkv7_backward_gn)
GN_PARAMS = ("gn_w", "gn_b", "r_k")
GN_GRADS = ("dgn_w", "dgn_b", "dr_k")


def run_gpu_gn(d, gp):
    """Forward + backward through the epilogue entry points; ``d["dy"]`` serves as do."""
    xs = [d[n] for n in INPUTS]
    o, y, sT, ck, fac = wkv7.forward_gn(*xs, gp["gn_w"], gp["gn_b"], gp["r_k"], s0=d.get("s0"), L=16)
    g = wkv7.backward_gn(*xs, ck, fac, y, d["dy"], gp["gn_w"], gp["r_k"], dsT=d.get("dsT"))
    torch.cuda.synchronize()
    wkv7.async_status()
    return {"o": o, "y": y, "sT": sT, "ckpt": ck, **g}


def oracle_head_gn(host, gp, b, h):
    """Oracle results of head (b, h) through recurrence + epilogue (B=H=1 shapes);
    the parameter gradients are this head's share of the sum over batch rows."""
    sl = {n: _head_input(host, n, b, h) for n in INPUTS + ("s0", "dy", "dsT")}
    p = {n: gp[n][h:h + 1] for n in GN_PARAMS}
    o, y, sT, ck = oracle.forward_gn(*(sl[n] for n in INPUTS), p["gn_w"], p["gn_b"], p["r_k"], s0=sl["s0"], L=16)
    res = {"o": o, "y": y, "sT": sT, "ckpt": ck}
    res.update(oracle.backward_gn(*(sl[n] for n in INPUTS), p["gn_w"], p["r_k"], sl["dy"], s0=sl["s0"], dsT=sl["dsT"]))
    return res


def check_heads_gn(host, gp, out, heads, B):
    """Every listed head element by element (o, y, sT, checkpoints at the forward
    bar; all gradients at the gradient bar), and the parameter gradients of every
    head index h that appears with all B batch rows, summed over them."""
    refs = oracle.per_head(lambda b, h: oracle_head_gn(host, gp, b, h), heads)
    worst = {}
    psum = {}
    for (b, h), ref in zip(heads, refs):
        got = gpu_head({k: v for k, v in out.items() if k not in GN_GRADS}, b, h)
        for k in ("o", "y", "sT", "ckpt"):
            e = max_rel(got[k], ref[k])
            assert e <= FWD_TOL, f"head ({b}, {h}) {k}: max err {e:.3e}"
            worst[k] = max(worst.get(k, 0.0), e)
        for k in GRADS + ("ds0",):
            e = grad_rel(got[k], ref[k])
            assert e <= GRAD_TOL, f"head ({b}, {h}) {k}: err {e:.3e}"
            worst[k] = max(worst.get(k, 0.0), e)
        for k in GN_GRADS:
            psum.setdefault(h, {}).setdefault(k, []).append(ref[k][0])
    for h, d in psum.items():
        if len(d["dgn_w"]) != B:
            continue
        for k in GN_GRADS:
            e = grad_rel(out[k][h].double().cpu().numpy(), np.sum(d[k], axis=0))
            assert e <= GRAD_TOL, f"h={h} {k}: err {e:.3e}"
            worst[k] = max(worst.get(k, 0.0), e)
    return worst
