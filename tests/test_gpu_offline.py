"""GPU: batched offline encoder over whole clips (vst_enc_offline) through the C ABI.

With the streaming mask (left = W = 750, right = 0) each clip's real rows equal, bit for
bit, the rows that streaming the clip through vst_enc_feed gives, whatever the padding
after them. With a right lookahead the rows match the fp64 oracle's (left, right) mask
within max|d| <= 2e-2 and mean|d| <= 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_kv_gb300 import synth, vst

pytestmark = pytest.mark.gpu

MAX_TOL = 2e-2
MEAN_TOL = 2e-3
H, D = 20, 64


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


def _clips(seed, B, T):
    """[B][T][H][D] bf16 q, k, v on the CPU (clip b from its own key stream)."""
    q = torch.stack([synth.frames(synth.tensor_key(seed, b, 0), 0, T, H, D, "cpu") for b in range(B)])
    k = torch.stack([synth.frames(synth.tensor_key(seed, b, 1), 0, T, H, D, "cpu") for b in range(B)])
    v = torch.stack([synth.frames(synth.tensor_key(seed, b, 2), 0, T, H, D, "cpu") for b in range(B)])
    return q, k, v


def _offline(module, dev, q, k, v, left, right):
    B, T = q.shape[0], q.shape[1]
    plan = vst.Offline(module, B, T)
    out = torch.empty((B, T, H, D), dtype=torch.bfloat16, device=dev)
    plan.run(q.to(dev), k.to(dev), v.to(dev), out, left, right)
    torch.cuda.synchronize()
    assert plan.check() == vst.OK
    plan.close()
    return out


def _stream(module, dev, q, k, v, chunk):
    """One clip [T][H][D] streamed in feeds of `chunk` frames: out [T][H][D]."""
    ctx = vst.Ctx(module)
    T = q.shape[0]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        vst.enc_feed(ctx.handle, qd[a:b], kd[a:b], vd[a:b], out[a:b])
    torch.cuda.synchronize()
    assert vst.ctx_check(ctx.handle) == vst.OK
    ctx.close()
    return out


def test_offline_equals_streaming(dev, enc_module):
    """Three clips right-padded to 2100 frames (real lengths 2100, 1300, 333): every real row
    equals the streamed clip's row, bit for bit (the streamed clips compact their ring)."""
    T, real = 2100, [2100, 1300, 333]
    q, k, v = _clips(41, 3, T)
    out = _offline(enc_module, dev, q, k, v, 750, 0)
    for b, n in enumerate(real):
        want = _stream(enc_module, dev, q[b, :n], k[b, :n], v[b, :n], 50 if b != 1 else 512)
        assert torch.equal(out[b, :n], want), b


@pytest.mark.parametrize("left,right", [(16, 4), (750, 4), (1, 1), (16, 0), (128, 129), (1000, 1000)])
def test_offline_lookahead_parity(dev, enc_module, left, right):
    """(left, right) masks on two clips of 300 frames (three query tiles, ragged tail)."""
    T = 300
    q, k, v = _clips(42, 2, T)
    out = _offline(enc_module, dev, q, k, v, left, right).float().cpu().double().numpy()
    for b in range(2):
        want = oracle.attention_lr(synth.bits(q[b]), synth.bits(k[b]), synth.bits(v[b]), left, right, threads=8)
        d = np.abs(out[b] - want)
        assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (b, d.max(), d.mean())


def test_offline_full_clips_sampled(dev, enc_module):
    """The offline workload the benchmark times, one layer: 4 clips x 4416 frames (seed 8,
    the same recipe) with left 750 and a right lookahead of 4. Rows at the clip ends, at
    query-tile edges and in the middle are compared with the oracle, each on its own window
    [i - 749, i + 3]."""
    seed, B, T, left, right = 8, 4, 4416, 750, 4
    mk = lambda n: torch.stack([synth.frames(synth.tensor_key(seed, b, 0, n), 0, T, H, D, dev) for b in range(B)])
    q, k, v = mk(0), mk(1), mk(2)
    plan = vst.Offline(enc_module, B, T)
    out = torch.empty_like(q)
    plan.run(q, k, v, out, left, right)
    torch.cuda.synchronize()
    assert plan.check() == vst.OK
    plan.close()
    got = out.float().cpu().double().numpy()
    for b in (0, 3):
        for i in (0, 1, 127, 128, 749, 750, 2000, 4351, 4352, 4412, 4415):
            a0, a1 = max(0, i - left + 1), min(T, i + right)  # keys of row i: [i - left + 1, i + right - 1]
            win = [synth.bits(synth.frames(synth.tensor_key(seed, b, 0, n), a0, a1 - a0, H, D, "cpu")) for n in range(3)]
            want = oracle.attention_lr(*win, left, right, pos0=a0, rows=(i - a0, i - a0 + 1))[0]
            d = np.abs(got[b, i] - want)
            assert np.isfinite(got[b, i]).all(), (b, i)
            assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (b, i, d.max(), d.mean())


def test_offline_layer_pattern(dev, enc_module):
    """The per-layer window pattern of the pages' Moonshine variant, (16, 4) (16, 4) (16, 0)
    (16, 0) (16, 4) (16, 4), one call per layer on one plan."""
    T, B = 200, 2
    plan = vst.Offline(enc_module, B, T)
    for layer, (left, right) in enumerate([(16, 4), (16, 4), (16, 0), (16, 0), (16, 4), (16, 4)]):
        q, k, v = _clips(50 + layer, B, T)
        out = torch.empty((B, T, H, D), dtype=torch.bfloat16, device=dev)
        plan.run(q.to(dev), k.to(dev), v.to(dev), out, left, right)
        torch.cuda.synchronize()
        got = out.float().cpu().double().numpy()
        for b in range(B):
            want = oracle.attention_lr(synth.bits(q[b]), synth.bits(k[b]), synth.bits(v[b]), left, right)
            d = np.abs(got[b] - want)
            assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (layer, b, d.max(), d.mean())
    assert plan.check() == vst.OK
    plan.close()


def test_offline_arguments(dev, enc_module):
    """Bad masks are refused with nothing enqueued; a decoder module has no offline plan."""
    plan = vst.Offline(enc_module, 1, 64)
    t = torch.zeros((1, 64, H, D), dtype=torch.bfloat16, device=dev)
    for left, right in ((0, 0), (16, -1)):
        with pytest.raises(RuntimeError):
            plan.run(t, t, t, t, left, right)
    plan.close()
    dec = vst.Module(vst.DEC)
    assert vst.offline_bytes(dec.handle, 1, 64) == 0
    with pytest.raises(RuntimeError):
        vst.Offline(dec, 1, 64)
    dec.close()
