"""Refusals of the streaming calls on live contexts. A call with a bad argument returns its
status before anything is enqueued, and every context it names is left as it was: its
bookkeeping is unchanged, vst_ctx_check reports no error, and its next good calls give the
bits that a context which never saw the bad call gives. (Checks that need no context run
on the CPU in test_host.py.)
"""
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


@pytest.fixture(scope="module")
def enc_module(dev):
    m = vst.Module(vst.ENC)
    yield m
    m.close()


@pytest.fixture(scope="module")
def dec_module(dev):
    m = vst.Module(vst.DEC)
    yield m
    m.close()


def _seq(seed, n, heads_q, heads_kv, d, dev):
    q = synth.frames(synth.tensor_key(seed, 0), 0, n, heads_q, d, "cpu").to(dev)
    k = synth.frames(synth.tensor_key(seed, 1), 0, n, heads_kv, d, "cpu").to(dev)
    v = synth.frames(synth.tensor_key(seed, 2), 0, n, heads_kv, d, "cpu").to(dev)
    return q, k, v


def _refused(fn, *args, **kw) -> int:
    with pytest.raises(vst.VstError) as e:
        fn(*args, **kw)
    return e.value.status


def _state(ctx):
    i = ctx.info()
    return (i.failed, i.n_kv, i.abs_base, i.abs_next, i.n_compactions)


def test_encoder_feed_refusals(dev, enc_module):
    T = 300
    q, k, v = _seq(41, T, 20, 20, 64, dev)
    out = torch.empty_like(q)
    a = vst.Ctx(enc_module)
    vst.enc_feed(a.handle, q[:100], k[:100], v[:100], out[:100])
    before = _state(a)
    raw = (q[100:].data_ptr(), k[100:].data_ptr(), v[100:].data_ptr(), out[100:].data_ptr())

    # the same context twice in one batch
    pair = [torch.stack([x[100:150], x[100:150]]).contiguous() for x in (q, k, v)]
    o2 = torch.empty_like(pair[0])
    assert _refused(vst.enc_feed_batch, [a.handle, a.handle], *pair, o2, 50) == vst.E_INVAL
    # contexts of two different modules in one batch
    other = vst.Module(vst.ENC)
    b = vst.Ctx(other)
    assert _refused(vst.enc_feed_batch, [a.handle, b.handle], *pair, o2, 50) == vst.E_INVAL
    # a negative row count, and pointers off the 16-byte alignment (raw pointers, past the
    # binding's size checks)
    assert _refused(vst.enc_feed, a.handle, *raw[:3], raw[3], n_new=-1) == vst.E_INVAL
    assert _refused(vst.enc_feed, a.handle, raw[0] + 2, *raw[1:3], raw[3], n_new=50) == vst.E_INVAL
    assert _refused(vst.enc_feed, a.handle, *raw[:3], raw[3] + 8, n_new=50) == vst.E_INVAL
    # positions past max_position
    assert _refused(vst.enc_feed, a.handle, *raw[:3], raw[3], n_new=int(enc_module.cfg.max_position)) == vst.E_INVAL
    # a decoder step on an encoder context
    qd = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device=dev)  # large enough for either kind
    assert _refused(vst.dec_step, [a.handle], qd, qd.clone(), qd.clone(), torch.empty_like(qd)) == vst.E_STATE
    torch.cuda.synchronize()
    assert _state(a) == before
    assert vst.ctx_check(a.handle) == vst.OK
    assert _state(b) == (0, 0, 0, 0, 0)
    b.close()
    other.close()

    # the refused calls left nothing behind: the rest of the stream equals a fresh context's
    vst.enc_feed(a.handle, q[100:], k[100:], v[100:], out[100:])
    ref = torch.empty_like(q)
    c = vst.Ctx(enc_module)
    vst.enc_feed(c.handle, q[:100], k[:100], v[:100], ref[:100])
    vst.enc_feed(c.handle, q[100:], k[100:], v[100:], ref[100:])
    torch.cuda.synchronize()
    assert vst.ctx_check(a.handle) == vst.OK
    assert _state(a) == _state(c)
    assert torch.equal(out, ref)
    a.close()
    c.close()


def test_decoder_step_refusals(dev, dec_module, enc_module):
    n = 40
    q, k, v = _seq(42, n, 32, 8, 128, dev)
    out = torch.empty_like(q)
    a = vst.Ctx(dec_module)
    for t in range(20):
        vst.dec_step([a.handle], q[t:t + 1], k[t:t + 1], v[t:t + 1], out[t:t + 1])
    before = _state(a)

    pair = [torch.cat([x[20:21], x[20:21]]).contiguous() for x in (q, k, v)]
    o2 = torch.empty_like(pair[0])
    # the same context twice in one step, and an empty context list
    assert _refused(vst.dec_step, [a.handle, a.handle], *pair, o2) == vst.E_INVAL
    assert _refused(vst.dec_step, [], *pair, o2) == vst.E_INVAL
    # an encoder context in a decoder step
    e = vst.Ctx(enc_module)
    assert _refused(vst.dec_step, [a.handle, e.handle], *pair, o2) == vst.E_INVAL
    e.close()
    # pointers off the 16-byte alignment
    assert _refused(vst.dec_step, [a.handle], q[20:].data_ptr() + 2, k[20:].data_ptr(), v[20:].data_ptr(),
                    out[20:].data_ptr()) == vst.E_INVAL
    torch.cuda.synchronize()
    assert _state(a) == before
    assert vst.ctx_check(a.handle) == vst.OK

    for t in range(20, n):
        vst.dec_step([a.handle], q[t:t + 1], k[t:t + 1], v[t:t + 1], out[t:t + 1])
    ref = torch.empty_like(q)
    c = vst.Ctx(dec_module)
    for t in range(n):
        vst.dec_step([c.handle], q[t:t + 1], k[t:t + 1], v[t:t + 1], ref[t:t + 1])
    torch.cuda.synchronize()
    assert vst.ctx_check(a.handle) == vst.OK
    assert _state(a) == _state(c)
    assert torch.equal(out, ref)
    a.close()
    c.close()
