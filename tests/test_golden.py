"""The hand-derived worked example of tests/golden/worked_example_t3.txt: every
value follows from the recurrence by hand (the derivation is in the file), so
it pins the oracle to something other than itself (state orientation, the
update's order, the sign of the rank-1 term, the decay axis and every
gradient), and the CUDA paths are checked against the same values."""
import os

import numpy as np
import pytest
import torch

from tests import parity

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_example_t3.txt")
N, T = 64, 3
INPUT_DEFAULTS = {"w": 0.25}


def load_fixture():
    inputs = {n: np.full((1, T, 1, N), INPUT_DEFAULTS.get(n, 0.0)) for n in ("r", "w", "k", "v", "a", "b", "dy")}
    expect = {}
    with open(FIXTURE) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            kind, name, i0, i1, val = line[0], line[1], int(line[2]), int(line[3]), float(line[4])
            if kind == "input":
                inputs[name][0, i0, 0, i1] = val
            elif kind == "expect":
                expect.setdefault(name, []).append((i0, i1, val))
            else:
                raise ValueError(f"unknown record {kind!r}")
    return inputs, expect


def dense(name, entries):
    shape = (1, 1, N, N) if name in ("sT", "ds0") else (1, T, 1, N)
    x = np.zeros(shape)
    for i0, i1, val in entries:
        if name in ("sT", "ds0"):
            x[0, 0, i0, i1] = val
        else:
            x[0, i0, 0, i1] = val
    return x


OUT_NAMES = ("y", "sT") + parity.GRADS + ("ds0",)


def test_fixture_is_complete():
    _, expect = load_fixture()
    assert set(expect) == set(OUT_NAMES)


def test_oracle_matches_the_worked_example():
    """Exact: every value of the example is a short sum of powers of two."""
    import oracle
    inputs, expect = load_fixture()
    ts = {n: torch.from_numpy(x.astype(np.float32)) for n, x in inputs.items()}
    y, sT, _ = oracle.forward(*(ts[n] for n in parity.INPUTS), L=16)
    got = {"y": np.asarray(y), "sT": np.asarray(sT)}
    got.update({k: np.asarray(v) for k, v in oracle.backward(*(ts[n] for n in parity.INPUTS), ts["dy"]).items()})
    for n in OUT_NAMES:
        np.testing.assert_array_equal(got[n], dense(n, expect[n]), err_msg=n)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,L", [("f32", 16), ("bf16", 16), ("f32", 1)])
def test_cuda_paths_match_the_worked_example(dtype, L):
    """The chunked path (L = 16) in fp32 and bf16 (every input value is exact in
    bf16) and the per-token path (L = 1), at the parity bars."""
    from rwkv_linear_attention_wkv7_gb300 import build, wkv7
    build()
    inputs, expect = load_fixture()
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    xs = [torch.from_numpy(inputs[n]).to(tdt).cuda() for n in parity.INPUTS]
    dy = torch.from_numpy(inputs["dy"]).float().cuda()
    y, sT, ck, *rest = wkv7.forward(*xs, L=L, want_factors=L == 16)
    g = wkv7.backward(*xs, ck, dy, L=L, factors=rest[0] if rest else None)
    torch.cuda.synchronize()
    wkv7.async_status()
    got = {"y": y, "sT": sT, **g}
    for n in OUT_NAMES:
        ref = dense(n, expect[n])
        err = np.abs(got[n].double().cpu().numpy() - ref).max() / np.abs(ref).max()
        bar = parity.FWD_TOL if n in ("y", "sT") else 1e-3
        assert err <= bar, (n, err)
