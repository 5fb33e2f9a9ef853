"""The chunked kernels' bounded waits, made to run out on purpose.

A test-only build of the library (-DWKV7_TEST_PHANTOM_TX) announces 16 bytes
more on one chunk's mbarrier than that chunk's copies deliver, so the wait for
that chunk can never complete -- a flag nothing sets; no copy is lost, no
address is wrong and nothing is left in flight.  The kernel must give up after
its time limit, leave its chunk loop, finish, and report the timeout through
wkv7_async_status; the context must stay usable (the regular library then
still matches the oracle).
"""
import time

import pytest
import torch

from rwkv_linear_attention_wkv7_gb300 import _build, synthetic, wkv7
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def phantom():
    _build.build()
    path = _build.build(variant="phantom_tx", extra_flags=["-DWKV7_TEST_PHANTOM_TX=1"])
    assert torch.cuda.is_available()
    return wkv7.load(path)


class _using:
    """Route the binding's calls to another build of the library for a while."""

    def __init__(self, lib):
        self.lib = lib

    def __enter__(self):
        self.saved = wkv7.lib()
        wkv7._lib = self.lib

    def __exit__(self, *exc):
        wkv7._lib = self.saved


def _timed(fn):
    torch.cuda.synchronize()
    t0 = time.monotonic()
    out = fn()
    torch.cuda.synchronize()
    return out, time.monotonic() - t0


def test_lost_copy_ends_the_forward_and_is_reported(phantom):
    spec = synthetic.WorkloadSpec("lost", 1, 64, 2, dtype="bf16", s0_std=0.1, seed=31)
    d, host = parity.inputs_on_device(spec)
    xs = [d[n] for n in parity.INPUTS]
    wkv7.async_status()  # start from a clear flag
    with _using(phantom):
        _, dt = _timed(lambda: wkv7.forward(*xs, s0=d["s0"], L=16))
        with pytest.raises(wkv7.WKV7Error) as e:
            wkv7.async_status()
        assert e.value.code == -2 and "ran out" in str(e.value)
        wkv7.async_status()  # reading the flag cleared it
    # one limit (0.5 s) for the wait that runs out and one for the final drain, per CTA, side by side
    assert dt < 5.0, dt
    out = parity.run_gpu(d, L=16)  # the regular build on the same context
    parity.check_heads(host, out, parity.all_heads(1, 2), L=16)


def test_lost_copy_ends_the_backward_and_is_reported(phantom):
    spec = synthetic.WorkloadSpec("lost", 1, 64, 2, dtype="f32", s0_std=0.1, with_dsT=True, seed=32)
    d, host = parity.inputs_on_device(spec)
    xs = [d[n] for n in parity.INPUTS]
    y, sT, ck, fac = wkv7.forward(*xs, s0=d["s0"], L=16, want_factors=True)
    wkv7.async_status()
    with _using(phantom):
        _, dt = _timed(lambda: wkv7.backward(*xs, ck, d["dy"], dsT=d["dsT"], L=16, factors=fac))
        with pytest.raises(wkv7.WKV7Error) as e:
            wkv7.async_status()
        assert e.value.code == -2
    assert dt < 5.0, dt
    out = parity.run_gpu(d, L=16)
    parity.check_heads(host, out, parity.all_heads(1, 2), L=16)
