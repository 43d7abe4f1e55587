"""GPU: failure detection without a fault.

Every kernel of the library bounds its device waits (TMA copies, MMA completions) by
%globaltimer time and, when one runs out, records a time-out in the context's error word
and winds down. Here a wait is made to run out on purpose -- an mbarrier that nothing
completes -- and the host reads the status through vst_ctx_check. No fault, trap or hang is
involved, and the context keeps working afterwards.
"""
import time

import pytest
import torch

from sliding_window_kv_gb300 import synth, vst

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    return torch.device("cuda:0")


def _feed(module, ctx, T, dev):
    q, k, v = (synth.frames(synth.tensor_key(61, 0, i), 0, T, 20, 64, "cpu").to(dev) for i in range(3))
    out = torch.empty_like(q)
    vst.enc_feed(ctx.handle, q, k, v, out)
    return out


def test_wait_timeout_reported_and_ctx_recovers(dev):
    m = vst.Module(vst.ENC)
    ctx = vst.Ctx(m)
    vst.ctx_selftest_wait(ctx.handle, True)
    assert vst.ctx_check(ctx.handle) == vst.OK

    t0 = time.perf_counter()
    vst.ctx_selftest_wait(ctx.handle, False)
    assert vst.ctx_check(ctx.handle) == vst.E_TIMEOUT
    waited = time.perf_counter() - t0
    assert 1.5 <= waited < 30.0, waited        # the wait's limit is 2 s of device time
    assert vst.ctx_check(ctx.handle) == vst.OK  # reading the status clears it

    # the context, the module and the device stay usable: a feed after the time-out gives
    # the bits a fresh context gives
    out = _feed(m, ctx, 300, dev)
    fresh = vst.Ctx(m)
    want = _feed(m, fresh, 300, dev)
    torch.cuda.synchronize()
    assert vst.ctx_check(ctx.handle) == vst.OK
    assert torch.equal(out, want)
    fresh.close()
    ctx.close()
    m.close()
