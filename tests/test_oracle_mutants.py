"""Plant plausible mistakes in a copy of the oracle's C source and check that
some pin catches each one (CPU only).  The copies are compiled into a
temporary directory; the oracle itself is never modified."""
import os

import pytest

import oracle
from tests.oracle_pins import ALL_PINS

# (name, text to replace, replacement, which occurrence (0-based))
MUTANTS = [
    ("sa uses b instead of a", "acc += S[i * N + j] * a[o + j];", "acc += S[i * N + j] * b[o + j];", 0),
    ("decay indexed by value row", "S[i * N + j] = S[i * N + j] * w[o + j]", "S[i * N + j] = S[i * N + j] * w[o + i]", 0),
    ("rank-1 term sign", "+ sa[i] * b[o + j] + v[o + i]", "- sa[i] * b[o + j] + v[o + i]", 0),
    ("v k^T transposed", "sa[i] * b[o + j] + v[o + i] * k[o + j];", "sa[i] * b[o + j] + v[o + j] * k[o + i];", 0),
    ("y reads with k", "acc += S[i * N + j] * r[o + j];", "acc += S[i * N + j] * k[o + j];", 0),
    ("first checkpoint skipped", "if (ckpt && t % L == 0) {", "if (ckpt && t % L == 0 && t > 0) {", 0),
    ("s0 ignored", "if (s0) memcpy(S, s0", "if (0) memcpy(S, s0", 0),
    ("bwd: dr from pre-update state", "acc += Sn[i * N + j] * dy[o + i];", "acc += Sp[i * N + j] * dy[o + i];", 0),
    ("bwd: carried gradient drops rank-1 term", "G[i * N + j] * w[o + j] + dsa[i] * a[o + j];", "G[i * N + j] * w[o + j];", 0),
    ("bwd: dw from post-update state", "acc_w += G[i * N + j] * Sp[i * N + j];", "acc_w += G[i * N + j] * Sn[i * N + j];", 0),
    ("bwd: db uses dsa", "acc_b += G[i * N + j] * sa[i];", "acc_b += G[i * N + j] * dsa[i];", 0),
    ("bwd: da transposed", "acc_a += Sp[i * N + j] * dsa[i];", "acc_a += Sp[j * N + i] * dsa[i];", 0),
    ("bwd: dv uses b", "acc_v += G[i * N + j] * k[o + j];", "acc_v += G[i * N + j] * b[o + j];", 0),
    ("bwd: dsT ignored", "if (dsT) memcpy(G,", "if (0) memcpy(G,", 0),
    ("bwd: dy r^T transposed", "G[i * N + j] += dy[o + i] * r[o + j];", "G[i * N + j] += dy[o + j] * r[o + i];", 0),
    ("decode: decay indexed by value row", "S[i * N + j] = S[i * N + j] * w[o + j]", "S[i * N + j] = S[i * N + j] * w[o + i]", 1),
]


def _replace_nth(text, old, new, n):
    pos = -1
    for _ in range(n + 1):
        pos = text.find(old, pos + 1)
        assert pos >= 0, f"mutation anchor not found: {old!r} (occurrence {n})"
    return text[:pos] + new + text[pos + len(old):]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_some_pin_catches(mutant, tmp_path):
    name, old, new, nth = mutant
    src = open(oracle.SOURCE).read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    c_path = os.path.join(tmp_path, "mutant.c")
    with open(c_path, "w") as f:
        f.write(mutated)
    so = oracle.compile_c(c_path, os.path.join(tmp_path, "libmutant.so"))
    orc = oracle.OracleLib(so)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake: {name}"


# Plausible mistakes in the fused producers and epilogues (Python side of the
# oracle), each swapped in for the real function; some fused pin must trip.
def _bad_producers(kind):
    real = oracle.producers

    def bad(w_pre, kk, avec):
        w, a, b, sigma = real(w_pre, kk, avec)
        kk64, avec64, wp = oracle._f64(kk), oracle._f64(avec), oracle._f64(w_pre)
        if kind == "decay coefficient doubled":
            w = w * w
        elif kind == "sigmoid dropped":
            w = oracle.np.exp(-oracle.DECAY * oracle.np.clip(wp, -50, 50))
        elif kind == "a = +kk":
            a = kk64
        elif kind == "b ignores avec":
            b = kk64
        elif kind == "b = avec":
            b = avec64
        return w, a, b, sigma
    return bad


def _bad_epilogue(kind):
    real = oracle.epilogue

    def bad(g, w, sigma, kk, avec):
        out = real(g, w, sigma, kk, avec)
        kk64, avec64 = oracle._f64(kk), oracle._f64(avec)
        if kind == "dw_pre without sigma(1 - sigma)":
            out["dw_pre"] = g["dw"] * w * (-oracle.DECAY)
        elif kind == "dkk sign of da":
            out["dkk"] = g["da"] + avec64 * g["db"]
        elif kind == "davec uses avec":
            out["davec"] = avec64 * g["db"]
        elif kind == "dkk drops db term":
            out["dkk"] = -g["da"]
        return out
    return bad


FUSED_MUTANTS = [("producers", k) for k in ("decay coefficient doubled", "sigmoid dropped", "a = +kk",
                                            "b ignores avec", "b = avec")] + \
                [("epilogue", k) for k in ("dw_pre without sigma(1 - sigma)", "dkk sign of da",
                                           "davec uses avec", "dkk drops db term")]


@pytest.mark.parametrize("mutant", FUSED_MUTANTS, ids=[m[1] for m in FUSED_MUTANTS])
def test_some_fused_pin_catches(mutant, monkeypatch):
    from tests.oracle_pins import FUSED_PINS
    where, kind = mutant
    if where == "producers":
        monkeypatch.setattr(oracle, "producers", _bad_producers(kind))
    else:
        monkeypatch.setattr(oracle, "epilogue", _bad_epilogue(kind))
    caught = []
    for pin in FUSED_PINS:
        try:
            pin(oracle.lib())
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no fused pin catches the planted mistake: {kind}"


# Plausible mistakes in the GroupNorm + bonus epilogue (Python side of the
# oracle), each swapped in for the real function; some epilogue pin must trip.
def _bad_gn(kind):
    real_f, real_b = oracle.gn_bonus, oracle.gn_bonus_backward
    np_ = oracle.np

    def fwd(y, r, k, v, gn_w, gn_b, r_k):
        y, r, k, v, gn_w, gn_b, r_k = map(oracle._f64, (y, r, k, v, gn_w, gn_b, r_k))
        n = y.shape[-1]
        mean = y.mean(axis=-1, keepdims=True)
        var = ((y - mean) ** 2).sum(axis=-1, keepdims=True) / (n - 1 if kind == "unbiased variance" else n)
        rstd = 1.0 / (np_.sqrt(var) + oracle.GN_EPS) if kind == "eps outside the root" else \
            1.0 / np_.sqrt(var + oracle.GN_EPS)
        g = (y - mean) * rstd * gn_w + gn_b
        if kind == "bonus from r twice":
            s = (r * r * r_k).sum(axis=-1, keepdims=True)
        elif kind == "bonus weight per value channel":
            return g + (r * k).sum(axis=-1, keepdims=True) * r_k * v, mean[..., 0], rstd[..., 0]
        else:
            s = (r * k * r_k).sum(axis=-1, keepdims=True)
        return g + s * v, mean[..., 0], rstd[..., 0]

    def bwd(y, r, k, v, gn_w, r_k, do):
        out = real_b(y, r, k, v, gn_w, r_k, do)
        y, r, k, v, gn_w, r_k, do = map(oracle._f64, (y, r, k, v, gn_w, r_k, do))
        n = y.shape[-1]
        mean = y.mean(axis=-1, keepdims=True)
        rstd = 1.0 / np_.sqrt(((y - mean) ** 2).mean(axis=-1, keepdims=True) + oracle.GN_EPS)
        xh = (y - mean) * rstd
        dn = do * gn_w
        ds = (do * v).sum(axis=-1, keepdims=True)
        if kind == "dy drops the mean of dn":
            out["dy"] = rstd * (dn - xh * (dn * xh).mean(axis=-1, keepdims=True))
        elif kind == "dy drops the projection on xh":
            out["dy"] = rstd * (dn - dn.mean(axis=-1, keepdims=True))
        elif kind == "bonus dr uses r":
            out["dr"] = ds * r * r_k
        elif kind == "d r_k misses k":
            out["dr_k"] = (ds * r).sum(axis=(0, 1))
        elif kind == "dgn_w from y":
            out["dgn_w"] = (do * y).sum(axis=(0, 1))
        elif kind == "dv without the bonus":
            out["dv"] = np_.zeros_like(out["dv"])
        return out

    fwd_kinds = ("unbiased variance", "eps outside the root", "bonus from r twice", "bonus weight per value channel")
    return (fwd if kind in fwd_kinds else real_f), (bwd if kind not in fwd_kinds else real_b)


GN_MUTANTS = ["unbiased variance", "eps outside the root", "bonus from r twice", "bonus weight per value channel",
              "dy drops the mean of dn", "dy drops the projection on xh", "bonus dr uses r", "d r_k misses k",
              "dgn_w from y", "dv without the bonus"]


@pytest.mark.parametrize("kind", GN_MUTANTS)
def test_some_gn_pin_catches(kind, monkeypatch):
    from tests.oracle_pins import GN_PINS
    f, b = _bad_gn(kind)
    monkeypatch.setattr(oracle, "gn_bonus", f)
    monkeypatch.setattr(oracle, "gn_bonus_backward", b)
    caught = []
    for pin in GN_PINS:
        try:
            pin(oracle.lib())
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no epilogue pin catches the planted mistake: {kind}"
