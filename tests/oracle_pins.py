"""Pins of the WKV7 oracle against what the pages and the mathematics fix.

Each ``pin_*`` takes an ``OracleLib`` and raises AssertionError when the
oracle disagrees with a fact that does not come from the oracle itself:
closed forms of special cases, exact invariants of the recurrence, central
finite differences and an automatic-differentiation adjoint.  The same pins
are run against deliberately broken copies of the oracle (see
``test_oracle_mutants.py``) to show that each plausible mistake trips one.

Notation (the "timemix.cu" page's WKV7 layout): token vectors [B][T][H][N],
state S[i][j] with i the value index and j the key index.
"""
from __future__ import annotations

import numpy as np

N = 64


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _decays(g, shape, lo=0.5, hi=1.0):
    return g.uniform(lo, hi, size=shape)


def _realistic(g, B, T, H):
    """Inputs shaped like an RWKV-7 time-mix block feeds them (a = -kk, b = kk*gate)."""
    shp = (B, T, H, N)
    r, k, v = (g.standard_normal(shp) for _ in range(3))
    kk = _unit(g.standard_normal(shp))
    gate = 1.0 / (1.0 + np.exp(-g.standard_normal(shp)))
    w = np.exp(-0.606531 / (1.0 + np.exp(-g.standard_normal(shp))))
    return dict(r=r, w=w, k=k, v=v, a=-kk, b=kk * gate)


def _close(got, want, rel, what):
    scale = max(1.0, float(np.abs(want).max()) if want.size else 1.0)
    err = float(np.abs(got - want).max()) if want.size else 0.0
    assert err <= rel * scale, f"{what}: max abs err {err:.3e} > {rel:.1e} x {scale:.3e}"


# ---------------------------------------------------------------- forward pins

def pin_linear_attention(orc):
    """w = 1, a = b = 0 reduces to causal linear attention:
    y_t = sum_{s<=t} v_s (k_s . r_t), and sT = sum_s v_s k_s^T."""
    g = _rng(1)
    B, T, H = 2, 13, 3
    r, k, v = (g.standard_normal((B, T, H, N)) for _ in range(3))
    one, zero = np.ones_like(r), np.zeros_like(r)
    y, sT, _ = orc.forward(r, one, k, v, zero, zero, L=4)
    scores = np.einsum("bthn,bshn->bhts", r, k) * np.tril(np.ones((T, T)))
    _close(y, np.einsum("bhts,bshn->bthn", scores, v), 1e-12, "linear attention y")
    _close(sT, np.einsum("bshi,bshj->bhij", v, k), 1e-12, "linear attention sT")


def pin_memoryless(orc):
    """w = 0, a = b = 0: every step forgets the past, y_t = v_t (k_t . r_t)."""
    g = _rng(2)
    B, T, H = 1, 7, 2
    r, k, v = (g.standard_normal((B, T, H, N)) for _ in range(3))
    s0 = g.standard_normal((B, H, N, N))
    zero = np.zeros_like(r)
    y, sT, _ = orc.forward(r, zero, k, v, zero, zero, s0=s0, L=3)
    _close(y, v * np.sum(k * r, axis=-1, keepdims=True), 1e-12, "memoryless y")
    _close(sT, np.einsum("bhi,bhj->bhij", v[:, -1], k[:, -1]), 1e-12, "memoryless sT")


def pin_decay_only(orc):
    """a = b = 0, per-key decay w: decayed linear attention with an initial state,
    y_t[i] = sum_j s0[i][j] prod_{u<=t} w_u[j] r_t[j]
           + sum_{s<=t} v_s[i] sum_j k_s[j] prod_{s<u<=t} w_u[j] r_t[j]."""
    g = _rng(3)
    B, T, H = 1, 9, 2
    r, k, v = (g.standard_normal((B, T, H, N)) for _ in range(3))
    w = _decays(g, (B, T, H, N), 0.3, 1.0)
    s0 = g.standard_normal((B, H, N, N))
    zero = np.zeros_like(r)
    y, _, _ = orc.forward(r, w, k, v, zero, zero, s0=s0, L=5)
    want = np.zeros_like(y)
    for bi in range(B):
        for h in range(H):
            for t in range(T):
                d0 = np.prod(w[bi, :t + 1, h], axis=0)
                acc = s0[bi, h] @ (d0 * r[bi, t, h])
                for s in range(t + 1):
                    d = np.prod(w[bi, s + 1:t + 1, h], axis=0)
                    acc = acc + v[bi, s, h] * np.dot(k[bi, s, h] * d, r[bi, t, h])
                want[bi, t, h] = acc
    _close(y, want, 1e-12, "decay-only y")


def pin_delta_rule_write(orc):
    """w = 1, a = -kk, b = kk, k = kk (unit): the step is the delta rule
    S <- S (I - kk kk^T) + v kk^T, after which S kk = v exactly.  Reading with
    r = kk therefore returns y_t = v_t whatever the earlier state."""
    g = _rng(4)
    B, T, H = 2, 6, 2
    kk = _unit(g.standard_normal((B, T, H, N)))
    v = g.standard_normal((B, T, H, N))
    s0 = g.standard_normal((B, H, N, N))
    y, sT, _ = orc.forward(kk, np.ones_like(kk), kk, v, -kk, kk, s0=s0, L=2)
    _close(y, v, 1e-12, "delta-rule read-back")
    _close(np.einsum("bhij,bhj->bhi", sT, kk[:, -1]), v[:, -1], 1e-12, "delta-rule sT kk")


def pin_projection_erases(orc):
    """w = 1, v = 0, a = -kk, b = kk: the transition I - kk kk^T is a projection,
    so the state forgets direction kk: S_t kk_t = 0 (read with r = kk)."""
    g = _rng(5)
    B, T, H = 1, 5, 3
    kk = _unit(g.standard_normal((B, T, H, N)))
    s0 = g.standard_normal((B, H, N, N))
    zero = np.zeros_like(kk)
    y, _, _ = orc.forward(kk, np.ones_like(kk), g.standard_normal(kk.shape), zero, -kk, kk,
                          s0=s0, L=2)
    _close(y, zero, 1e-12, "projection erases kk")


def pin_rank1_orientation(orc):
    """w = 1, v = 0, one step: S1 = S0 (I + a b^T).  For r orthogonal to b the
    step leaves the read unchanged, y = S0 r; the transposed transition
    S0 (I + b a^T) would add (S0 b)(a . r)."""
    g = _rng(6)
    B, H = 2, 3
    a = g.standard_normal((B, 1, H, N))
    b = g.standard_normal((B, 1, H, N))
    r = g.standard_normal((B, 1, H, N))
    r = r - b * (np.sum(r * b, -1, keepdims=True) / np.sum(b * b, -1, keepdims=True))
    s0 = g.standard_normal((B, H, N, N))
    y, _, _ = orc.forward(r, np.ones_like(r), g.standard_normal(r.shape), np.zeros_like(r),
                          a, b, s0=s0, L=1)
    _close(y[:, 0], np.einsum("bhij,bhj->bhi", s0, r[:, 0]), 1e-12, "rank-1 orientation")


def pin_empty_sequence(orc):
    """T = 0: no token, so sT = s0, no checkpoint, ds0 = dsT and no gradients."""
    g = _rng(7)
    s0 = g.standard_normal((2, 3, N, N))
    dsT = g.standard_normal((2, 3, N, N))
    e = np.zeros((2, 0, 3, N))
    y, sT, ck = orc.forward(e, e, e, e, e, e, s0=s0, L=4)
    assert y.shape == (2, 0, 3, N) and ck.shape == (2, 3, 0, N, N)
    _close(sT, s0, 0.0, "T=0 sT")
    gr = orc.backward(e, e, e, e, e, e, e, s0=s0, dsT=dsT)
    _close(gr["ds0"], dsT, 0.0, "T=0 ds0")


# --------------------------------------------------------- structural invariants

def pin_checkpoints_are_prefix_states(orc):
    """ckpt[c] is the state before token c*L, i.e. the final state of the first
    c*L tokens (ckpt[0] = s0), including a ragged last interval."""
    g = _rng(8)
    B, T, H, L = 1, 11, 2, 4
    x = _realistic(g, B, T, H)
    s0 = 0.1 * g.standard_normal((B, H, N, N))
    _, _, ck = orc.forward(**x, s0=s0, L=L)
    assert ck.shape == (B, H, 3, N, N)
    for c in range(3):
        pre = {n: x[n][:, :c * L] for n in x}
        _, s_c, _ = orc.forward(**pre, s0=s0, L=L)
        _close(ck[:, :, c], s_c, 0.0, f"checkpoint {c}")


def pin_split_sequence(orc):
    """Running T1 tokens, then T2 tokens from the carried state, equals one
    T1+T2 call (same operation order, so bit for bit)."""
    g = _rng(9)
    B, T, H, T1 = 2, 10, 2, 3
    x = _realistic(g, B, T, H)
    s0 = 0.1 * g.standard_normal((B, H, N, N))
    y, sT, _ = orc.forward(**x, s0=s0, L=4)
    y1, s1, _ = orc.forward(**{n: x[n][:, :T1] for n in x}, s0=s0, L=4)
    y2, s2, _ = orc.forward(**{n: x[n][:, T1:] for n in x}, s0=s1, L=4)
    _close(np.concatenate([y1, y2], axis=1), y, 0.0, "split y")
    _close(s2, sT, 0.0, "split sT")


def pin_decode_is_streaming(orc):
    """Feeding the tokens one at a time through the decode step (state updated in
    place, the streaming-inference use) reproduces the sequence call bit for bit."""
    g = _rng(10)
    B, T, H = 2, 5, 3
    x = _realistic(g, B, T, H)
    s0 = 0.1 * g.standard_normal((B, H, N, N))
    y, sT, _ = orc.forward(**x, s0=s0, L=2)
    st = s0.copy()
    for t in range(T):
        yt, st = orc.decode_step(*(x[n][:, t] for n in ("r", "w", "k", "v", "a", "b")), st)
        _close(yt, y[:, t], 0.0, f"decode token {t}")
    _close(st, sT, 0.0, "decode state")


def pin_linear_in_state_and_values(orc):
    """For fixed r, w, k, a, b the recurrence is linear in (s0, v) jointly:
    y(s0, v) = y(s0, 0) + y(0, v)."""
    g = _rng(11)
    B, T, H = 1, 8, 2
    x = _realistic(g, B, T, H)
    s0 = g.standard_normal((B, H, N, N))
    y, sT, _ = orc.forward(**x, s0=s0, L=3)
    y_s, sT_s, _ = orc.forward(**{**x, "v": np.zeros_like(x["v"])}, s0=s0, L=3)
    y_v, sT_v, _ = orc.forward(**x, s0=None, L=3)
    _close(y, y_s + y_v, 1e-12, "linearity y")
    _close(sT, sT_s + sT_v, 1e-12, "linearity sT")


# ----------------------------------------------------------------- backward pins

def _loss(orc, x, s0, dy, dsT):
    y, sT, _ = orc.forward(**x, s0=s0, L=4, want_ckpt=False)
    return float(np.sum(y * dy) + np.sum(sT * dsT))


def pin_worked_example(orc):
    """The hand-derived worked example of tests/golden/worked_example_t3.txt
    (its derivation is in the file): y, sT and every gradient, exactly."""
    from tests.test_golden import OUT_NAMES, dense, load_fixture
    inputs, expect = load_fixture()
    x = {n: inputs[n] for n in ("r", "w", "k", "v", "a", "b")}
    y, sT, _ = orc.forward(**x, L=16)
    got = {"y": y, "sT": sT, **orc.backward(**x, dy=inputs["dy"])}
    for n in OUT_NAMES:
        want = dense(n, expect[n])
        assert np.array_equal(np.asarray(got[n]), want), f"worked example {n}: max diff {np.abs(got[n] - want).max():.3e}"


def pin_adjoint_identity(orc):
    """y and sT are linear in (s0, v), so for any direction (u0, uv):
    <y(u0, uv), dy> + <sT(u0, uv), dsT> = <u0, ds0> + <uv, dv>."""
    g = _rng(12)
    B, T, H = 1, 9, 2
    x = _realistic(g, B, T, H)
    dy = g.standard_normal(x["r"].shape)
    dsT = g.standard_normal((B, H, N, N))
    gr = orc.backward(**x, dy=dy, s0=g.standard_normal((B, H, N, N)), dsT=dsT)
    u0 = g.standard_normal((B, H, N, N))
    uv = g.standard_normal(x["v"].shape)
    lhs = _loss(orc, {**x, "v": uv}, u0, dy, dsT)
    rhs = float(np.sum(u0 * gr["ds0"]) + np.sum(uv * gr["dv"]))
    assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs)), f"adjoint {lhs!r} vs {rhs!r}"


def pin_finite_differences(orc):
    """Central finite differences in float64 on a tiny problem: every gradient
    (dr, dw, dk, dv, da, db, ds0) at sampled coordinates, relative error < 1e-6
    (the bar the pages set for f64 gradchecks is 1e-3)."""
    g = _rng(13)
    B, T, H = 1, 6, 1
    x = _realistic(g, B, T, H)
    s0 = 0.5 * g.standard_normal((B, H, N, N))
    dy = g.standard_normal(x["r"].shape)
    dsT = g.standard_normal((B, H, N, N))
    gr = orc.backward(**x, dy=dy, s0=s0, dsT=dsT)
    eps = 1e-6
    for name in ("r", "w", "k", "v", "a", "b", "s0"):
        base = s0 if name == "s0" else x[name]
        grad = gr["d" + name]
        scale = float(np.abs(grad).max())
        for idx in [tuple(int(g.integers(0, s)) for s in base.shape) for _ in range(10)]:
            def loss_at(delta):
                pert = base.copy()
                pert[idx] += delta
                if name == "s0":
                    return _loss(orc, x, pert, dy, dsT)
                return _loss(orc, {**x, name: pert}, s0, dy, dsT)
            fd = (loss_at(eps) - loss_at(-eps)) / (2 * eps)
            err = abs(fd - grad[idx]) / max(abs(grad[idx]), 1e-3 * scale)
            assert err < 1e-6, f"d{name}{idx}: fd {fd:.9e} vs {grad[idx]:.9e} (rel {err:.2e})"


def pin_autograd_adjoint(orc):
    """The hand-written adjoint equals the one torch's autograd derives (float64)
    from the recurrence written with the transition matrix P_t = diag(w_t) + a_t b_t^T:
    S_t = S_{t-1} P_t + v_t k_t^T, y_t = S_t r_t."""
    import torch
    g = _rng(14)
    B, T, H = 1, 7, 2
    x = _realistic(g, B, T, H)
    s0 = 0.3 * g.standard_normal((B, H, N, N))
    dy = g.standard_normal(x["r"].shape)
    dsT = g.standard_normal((B, H, N, N))
    gr = orc.backward(**x, dy=dy, s0=s0, dsT=dsT)
    tx = {n: torch.tensor(x[n], requires_grad=True) for n in x}
    ts0 = torch.tensor(s0, requires_grad=True)
    S = ts0
    ys = []
    for t in range(T):
        P = torch.diag_embed(tx["w"][:, t]) + tx["a"][:, t, :, :, None] * tx["b"][:, t, :, None, :]
        S = S @ P + tx["v"][:, t, :, :, None] * tx["k"][:, t, :, None, :]
        ys.append((S @ tx["r"][:, t, :, :, None])[..., 0])
    loss = (torch.stack(ys, 1) * torch.tensor(dy)).sum() + (S * torch.tensor(dsT)).sum()
    loss.backward()
    for n in tx:
        _close(gr["d" + n], tx[n].grad.numpy(), 1e-11, f"autograd d{n}")
    _close(gr["ds0"], ts0.grad.numpy(), 1e-11, "autograd ds0")


# ------------------------------------------- fused producers and epilogues
# The fused entry points take (r, w_pre, k, v, kk, avec): w = exp(-0.606531 sigmoid(w_pre)),
# a = -kk, b = kk * avec ("timemix.cu" page, k_decay and k_composites).

def _fused_inputs(g, B, T, H):
    shp = (B, T, H, N)
    r, k, v, w_pre = (g.standard_normal(shp) for _ in range(4))
    kk = _unit(g.standard_normal(shp))
    avec = 1.0 / (1.0 + np.exp(-g.standard_normal(shp)))
    return dict(r=r, w_pre=w_pre, k=k, v=v, kk=kk, avec=avec)


def pin_fused_constant_decay(orc):
    """kk = 0 removes the rank-1 term; a constant pre-activation gives one decay
    c for every key: sigmoid(0) = 1/2 gives c = exp(-0.606531/2), a saturated
    sigmoid c = exp(-0.606531).  Then
    y_t = c^{t+1} s0 r_t + sum_{s<=t} c^{t-s} v_s (k_s . r_t)."""
    g = _rng(21)
    B, T, H = 1, 8, 2
    x = _fused_inputs(g, B, T, H)
    x["kk"] = np.zeros_like(x["kk"])
    s0 = g.standard_normal((B, H, N, N))
    for wp, c in ((0.0, np.exp(-0.606531 / 2)), (60.0, np.exp(-0.606531))):
        y, _, _ = orc.forward_fused(**{**x, "w_pre": np.full_like(x["r"], wp)}, s0=s0, L=3)
        r, k, v = x["r"], x["k"], x["v"]
        want = np.zeros_like(y)
        for t in range(T):
            acc = c ** (t + 1) * np.einsum("bhij,bhj->bhi", s0, r[:, t])
            for s_ in range(t + 1):
                acc = acc + c ** (t - s_) * v[:, s_] * np.sum(k[:, s_] * r[:, t], -1, keepdims=True)
            want[:, t] = acc
        _close(y, want, 1e-12, f"fused constant decay at w_pre={wp}")


def pin_fused_delta_rule(orc):
    """A very negative pre-activation gives w = 1.  With avec = 1 and k = kk
    (unit) the step is the delta rule S <- S (I - kk kk^T) + v kk^T, so reading
    with r = kk returns v_t; with avec = 0 the rank-1 term vanishes and the
    read is causal linear attention."""
    g = _rng(22)
    B, T, H = 2, 6, 2
    kk = _unit(g.standard_normal((B, T, H, N)))
    v = g.standard_normal((B, T, H, N))
    s0 = g.standard_normal((B, H, N, N))
    w_pre = np.full_like(kk, -800.0)
    y, _, _ = orc.forward_fused(kk, w_pre, kk, v, kk, np.ones_like(kk), s0=s0, L=2)
    _close(y, v, 1e-12, "fused delta-rule read-back")
    r, k = g.standard_normal(kk.shape), g.standard_normal(kk.shape)
    y0, _, _ = orc.forward_fused(r, w_pre, k, v, kk, np.zeros_like(kk), L=2)
    scores = np.einsum("bthn,bshn->bhts", r, k) * np.tril(np.ones((T, T)))
    _close(y0, np.einsum("bhts,bshn->bthn", scores, v), 1e-12, "fused avec = 0 is linear attention")


def _fused_loss(orc, x, s0, dy, dsT):
    y, sT, _ = orc.forward_fused(**x, s0=s0, L=4, want_ckpt=False)
    return float(np.sum(y * dy) + np.sum(sT * dsT))


def pin_fused_finite_differences(orc):
    """Central finite differences in float64 of the fused forward: every fused
    gradient (dr, dw_pre, dk, dv, dkk, davec, ds0) at sampled coordinates,
    relative error < 1e-5 (the difference quotient's rounding noise is about
    1e-7 here; a wrong epilogue term is off by order 1)."""
    g = _rng(23)
    B, T, H = 1, 5, 1
    x = _fused_inputs(g, B, T, H)
    s0 = 0.5 * g.standard_normal((B, H, N, N))
    dy = g.standard_normal(x["r"].shape)
    dsT = g.standard_normal((B, H, N, N))
    gr = orc.backward_fused(**x, dy=dy, s0=s0, dsT=dsT)
    eps = 1e-6
    for name in ("r", "w_pre", "k", "v", "kk", "avec", "s0"):
        base = s0 if name == "s0" else x[name]
        grad = gr["d" + name]
        scale = float(np.abs(grad).max())
        for idx in [tuple(int(g.integers(0, s)) for s in base.shape) for _ in range(8)]:
            def loss_at(delta):
                pert = base.copy()
                pert[idx] += delta
                if name == "s0":
                    return _fused_loss(orc, x, pert, dy, dsT)
                return _fused_loss(orc, {**x, name: pert}, s0, dy, dsT)
            fd = (loss_at(eps) - loss_at(-eps)) / (2 * eps)
            err = abs(fd - grad[idx]) / max(abs(grad[idx]), 1e-3 * scale)
            assert err < 1e-5, f"d{name}{idx}: fd {fd:.9e} vs {grad[idx]:.9e} (rel {err:.2e})"


FUSED_PINS = [pin_fused_constant_decay, pin_fused_delta_rule, pin_fused_finite_differences]


# ------------------------------------------- GroupNorm + bonus output epilogue
# ("timemix.cu" page: k_groupnorm, k_bonus and their backward kernels).  These
# pins take the module-level oracle functions, so that planted mistakes can be
# swapped in for them (test_oracle_mutants.py).

def _gn_inputs(g, B, T, H):
    shp = (B, T, H, N)
    y, r, k, v = (g.standard_normal(shp) for _ in range(4))
    gn_w, gn_b, r_k = (g.standard_normal((H, N)) for _ in range(3))
    return dict(y=y, r=r, k=k, v=v, gn_w=gn_w, gn_b=gn_b, r_k=r_k)


def pin_gn_library_groupnorm(orc):
    """With r_k = 0 the epilogue is a GroupNorm with one group of N channels
    per head over the C = H N channels of a token: torch's own group_norm in
    float64 (eps 64e-5) gives the same output, and torch autograd through it
    gives the same dy, dgn_w and dgn_b."""
    import torch
    import oracle
    g = _rng(31)
    B, T, H = 2, 5, 3
    x = _gn_inputs(g, B, T, H)
    zero = np.zeros((H, N))
    o, _, _ = oracle.gn_bonus(x["y"], x["r"], x["k"], x["v"], x["gn_w"], x["gn_b"], zero)
    y = torch.tensor(x["y"].reshape(B * T, H * N), requires_grad=True)
    w = torch.tensor(x["gn_w"].reshape(-1), requires_grad=True)
    b = torch.tensor(x["gn_b"].reshape(-1), requires_grad=True)
    ref = torch.nn.functional.group_norm(y, H, w, b, eps=64e-5)
    _close(o, ref.detach().numpy().reshape(B, T, H, N), 1e-12, "GroupNorm output")
    do = g.standard_normal((B, T, H, N))
    (ref * torch.tensor(do.reshape(B * T, H * N))).sum().backward()
    e = oracle.gn_bonus_backward(x["y"], x["r"], x["k"], x["v"], x["gn_w"], zero, do)
    _close(e["dy"], y.grad.numpy().reshape(B, T, H, N), 1e-12, "GroupNorm dy")
    _close(e["dgn_w"], w.grad.numpy().reshape(H, N), 1e-12, "GroupNorm dgn_w")
    _close(e["dgn_b"], b.grad.numpy().reshape(H, N), 1e-12, "GroupNorm dgn_b")


def pin_gn_standardised_input(orc):
    """y = a z + c with z of exactly zero mean and unit (biased) variance over
    the head: with gn_w = 1, gn_b = 0, r_k = 0 the output is z a / sqrt(a^2 + 64e-5),
    whatever c; and with y constant over the head (a = 0) it is gn_b."""
    import oracle
    g = _rng(32)
    B, T, H = 1, 6, 2
    x = _gn_inputs(g, B, T, H)
    z = g.standard_normal((B, T, H, N))
    z = z - z.mean(axis=-1, keepdims=True)
    z = z / np.sqrt((z ** 2).mean(axis=-1, keepdims=True))
    a = g.uniform(0.05, 3.0, size=(B, T, H, 1))
    c = g.standard_normal((B, T, H, 1)) * 5
    one, zero = np.ones((H, N)), np.zeros((H, N))
    o, _, _ = oracle.gn_bonus(a * z + c, x["r"], x["k"], x["v"], one, zero, zero)
    _close(o, z * a / np.sqrt(a ** 2 + 64e-5), 1e-12, "standardised input")
    o, _, _ = oracle.gn_bonus(np.broadcast_to(c, z.shape), x["r"], x["k"], x["v"], x["gn_w"], x["gn_b"], zero)
    _close(o, np.broadcast_to(x["gn_b"], o.shape), 1e-12, "constant input gives the bias")


def pin_gn_bonus_one_channel(orc):
    """A bonus weight on one channel m only (r_k = e_m) adds r_m k_m v to the
    GroupNorm output: the bonus is the r, k product of that channel scaling
    the whole value vector."""
    import oracle
    g = _rng(33)
    B, T, H = 2, 4, 3
    x = _gn_inputs(g, B, T, H)
    zero = np.zeros((H, N))
    base, _, _ = oracle.gn_bonus(x["y"], x["r"], x["k"], x["v"], x["gn_w"], x["gn_b"], zero)
    for m in (0, 17, 63):
        rk = np.zeros((H, N))
        rk[:, m] = 1.0
        o, _, _ = oracle.gn_bonus(x["y"], x["r"], x["k"], x["v"], x["gn_w"], x["gn_b"], rk)
        want = base + (x["r"][..., m] * x["k"][..., m])[..., None] * x["v"]
        _close(o, want, 1e-12, f"bonus on channel {m}")


def pin_gn_finite_differences(orc):
    """Central finite differences in float64 of sum(o do) through the
    epilogue: dy, dr, dk, dv, dgn_w, dgn_b, dr_k at sampled coordinates,
    relative error < 1e-6."""
    import oracle
    g = _rng(34)
    B, T, H = 2, 3, 2
    x = _gn_inputs(g, B, T, H)
    do = g.standard_normal((B, T, H, N))
    e = oracle.gn_bonus_backward(x["y"], x["r"], x["k"], x["v"], x["gn_w"], x["r_k"], do)

    def loss(xx):
        o, _, _ = oracle.gn_bonus(xx["y"], xx["r"], xx["k"], xx["v"], xx["gn_w"], xx["gn_b"], xx["r_k"])
        return float(np.sum(o * do))
    eps = 1e-6
    for name in ("y", "r", "k", "v", "gn_w", "gn_b", "r_k"):
        grad = e["d" + name]
        scale = float(np.abs(grad).max())
        for idx in [tuple(int(g.integers(0, s)) for s in x[name].shape) for _ in range(6)]:
            def at(delta):
                pert = x[name].copy()
                pert[idx] += delta
                return loss({**x, name: pert})
            fd = (at(eps) - at(-eps)) / (2 * eps)
            err = abs(fd - grad[idx]) / max(abs(grad[idx]), 1e-3 * scale, 1e-300)
            assert err < 1e-6, f"d{name}{idx}: fd {fd:.9e} vs {grad[idx]:.9e} (rel {err:.2e})"


def pin_gn_composite_finite_differences(orc):
    """The recurrence followed by the epilogue: central finite differences of
    sum(o do) + sum(sT dsT) for r, w, k, v, a, b, s0 and the three epilogue
    weights against backward_gn (which adds the bonus's own dr, dk, dv to the
    recurrence's), relative error < 1e-5."""
    g = _rng(35)
    B, T, H = 1, 5, 1
    x = _realistic(g, B, T, H)
    p = {n: g.standard_normal((H, N)) for n in ("gn_w", "gn_b", "r_k")}
    s0 = 0.5 * g.standard_normal((B, H, N, N))
    do = g.standard_normal((B, T, H, N))
    dsT = g.standard_normal((B, H, N, N))
    gr = orc.backward_gn(*(x[n] for n in "rwkvab"), p["gn_w"], p["r_k"], do, s0=s0, dsT=dsT)

    def loss(xx, pp, ss):
        o, _, sT, _ = orc.forward_gn(*(xx[n] for n in "rwkvab"), pp["gn_w"], pp["gn_b"], pp["r_k"], s0=ss, L=4,
                                     want_ckpt=False)
        return float(np.sum(o * do) + np.sum(sT * dsT))
    eps = 1e-6
    for name in ("r", "w", "k", "v", "a", "b", "s0", "gn_w", "gn_b", "r_k"):
        base = s0 if name == "s0" else (p[name] if name in p else x[name])
        grad = gr["d" + name]
        scale = float(np.abs(grad).max())
        for idx in [tuple(int(g.integers(0, s)) for s in base.shape) for _ in range(4)]:
            def at(delta):
                pert = base.copy()
                pert[idx] += delta
                if name == "s0":
                    return loss(x, p, pert)
                if name in p:
                    return loss(x, {**p, name: pert}, s0)
                return loss({**x, name: pert}, p, s0)
            fd = (at(eps) - at(-eps)) / (2 * eps)
            err = abs(fd - grad[idx]) / max(abs(grad[idx]), 1e-3 * scale, 1e-300)
            assert err < 1e-5, f"d{name}{idx}: fd {fd:.9e} vs {grad[idx]:.9e} (rel {err:.2e})"


GN_PINS = [pin_gn_library_groupnorm, pin_gn_standardised_input, pin_gn_bonus_one_channel, pin_gn_finite_differences,
           pin_gn_composite_finite_differences]

ALL_PINS = [
    pin_linear_attention, pin_memoryless, pin_decay_only, pin_delta_rule_write,
    pin_projection_erases, pin_rank1_orientation, pin_empty_sequence,
    pin_checkpoints_are_prefix_states, pin_split_sequence, pin_decode_is_streaming,
    pin_linear_in_state_and_values, pin_adjoint_identity, pin_finite_differences,
    pin_autograd_adjoint, pin_worked_example,
] + FUSED_PINS + GN_PINS
