"""GPU: decoder prefill (vst_dec_prefill) through the C ABI.

A prefill of n tokens must give, bit for bit, what n successive one-token decoder steps
give (same ring bytes afterwards too), and match the fp64 oracle within max|d| <= 2e-2 and
mean|d| <= 2e-3. The cases cover the pages' 39-token prompt, several 64-token chunks, a
prefill that crosses the point where a ring of R = W slots starts evicting (chunks shrink to
one token there), and a ring a little larger than the window (chunks stay 64 long across
the wrap).
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_kv_gb300 import synth, vst

pytestmark = pytest.mark.gpu

MAX_TOL = 2e-2
MEAN_TOL = 2e-3
W = 8192


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def dec_module(dev):
    m = vst.Module(vst.DEC)
    yield m
    m.close()


def _dec_seq(seed, stream, n_tok, first=0):
    q = synth.frames(synth.tensor_key(seed, stream, 0, 0), first, n_tok, 32, 128, "cpu")
    k = synth.frames(synth.tensor_key(seed, stream, 0, 1), first, n_tok, 8, 128, "cpu")
    v = synth.frames(synth.tensor_key(seed, stream, 0, 2), first, n_tok, 8, 128, "cpu")
    return q, k, v


class _Ctx:
    """A decoder ctx on caller-owned memory, so the rings can be compared."""

    def __init__(self, module, dev):
        nbytes = vst.ctx_bytes(module.handle)
        self.mem = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.handle = vst.ctx_create(module.handle, self.mem.data_ptr(), nbytes)
        info = vst.ctx_info_get(self.handle)
        cfg = module.cfg
        n = cfg.n_kv_heads * cfg.ring_slots * cfg.head_dim * 2
        base = self.mem.data_ptr()
        self.k_ring = self.mem[info.k_ring - base:info.k_ring - base + n]
        self.v_ring = self.mem[info.v_ring - base:info.v_ring - base + n]

    def close(self):
        vst.ctx_destroy(self.handle)


def _steps(module, dev, q, k, v, fill, n):
    """`fill` tokens appended, then n one-token steps: (out [n][32][128], ctx)."""
    ctx = _Ctx(module, dev)
    if fill:
        vst.dec_append(ctx.handle, k[:fill].to(dev), v[:fill].to(dev))
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty((n, 32, 128), dtype=torch.bfloat16, device=dev)
    for s in range(n):
        t = fill + s
        vst.dec_step([ctx.handle], qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], out[s:s + 1])
    torch.cuda.synchronize()
    assert vst.ctx_check(ctx.handle) == vst.OK
    return out, ctx


def _prefill(module, dev, q, k, v, fill, n, pieces=None):
    """`fill` tokens appended, then tokens [fill, fill + n) by vst_dec_prefill calls of the
    given sizes (one call by default): (out, ctx)."""
    ctx = _Ctx(module, dev)
    if fill:
        vst.dec_append(ctx.handle, k[:fill].to(dev), v[:fill].to(dev))
    out = torch.empty((n, 32, 128), dtype=torch.bfloat16, device=dev)
    t = 0
    for p in (pieces or [n]):
        a, b = fill + t, fill + t + p
        vst.dec_prefill(ctx.handle, q[a:b].to(dev), k[a:b].to(dev), v[a:b].to(dev), out[t:t + p])
        t += p
    torch.cuda.synchronize()
    assert vst.ctx_check(ctx.handle) == vst.OK
    assert vst.ctx_info_get(ctx.handle).abs_next == fill + n
    return out, ctx


def _oracle_rows(q, k, v, rows):
    qb, kb, vb = synth.bits(q), synth.bits(k), synth.bits(v)
    return [oracle.attention_row(qb[i], kb[max(0, i - W + 1):i + 1], vb[max(0, i - W + 1):i + 1], i, W)
            for i in rows]


def _same(a_out, a_ctx, b_out, b_ctx):
    assert torch.equal(a_out, b_out)
    assert torch.equal(a_ctx.k_ring, b_ctx.k_ring)
    assert torch.equal(a_ctx.v_ring, b_ctx.v_ring)


def test_prefill_prompt_39(dev, dec_module):
    """The pages' prompt length: 39 tokens on an empty cache, one launch."""
    q, k, v = _dec_seq(21, 0, 39)
    out, ctx = _prefill(dec_module, dev, q, k, v, 0, 39)
    ref, rctx = _steps(dec_module, dev, q, k, v, 0, 39)
    _same(out, ctx, ref, rctx)
    want = oracle.attention(synth.bits(q), synth.bits(k), synth.bits(v), window=W, threads=8)
    d = np.abs(out.float().cpu().double().numpy() - want)
    assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (d.max(), d.mean())
    ctx.close()
    rctx.close()


@pytest.mark.parametrize("fill,n,pieces", [(0, 1, None), (5, 150, None), (300, 200, [1, 63, 64, 72])])
def test_prefill_equals_steps(dev, dec_module, fill, n, pieces):
    """Chunks of 64 and ragged calls: the same bits as one-token steps, then more steps
    after the prefill continue identically."""
    q, k, v = _dec_seq(22, fill, fill + n + 3)
    out, ctx = _prefill(dec_module, dev, q, k, v, fill, n, pieces)
    ref, rctx = _steps(dec_module, dev, q, k, v, fill, n)
    _same(out, ctx, ref, rctx)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1 = torch.empty((1, 32, 128), dtype=torch.bfloat16, device=dev)
    o2 = torch.empty_like(o1)
    for t in range(fill + n, fill + n + 3):
        vst.dec_step([ctx.handle], qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], o1)
        vst.dec_step([rctx.handle], qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], o2)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    rows = [fill, fill + n // 2, fill + n - 1]
    got = out.float().cpu().double().numpy()
    for i, want in zip(rows, _oracle_rows(q, k, v, rows)):
        d = np.abs(got[i - fill] - want)
        assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (i, d.max(), d.mean())
    ctx.close()
    rctx.close()


def test_prefill_across_eviction(dev, dec_module):
    """R = W = 8192: tokens below position 8192 go in chunks, later ones one per launch
    (each evicts a key the chunk's earlier tokens still see)."""
    fill, n = 8100, 160
    q, k, v = _dec_seq(23, 0, fill + n)
    out, ctx = _prefill(dec_module, dev, q, k, v, fill, n)
    ref, rctx = _steps(dec_module, dev, q, k, v, fill, n)
    _same(out, ctx, ref, rctx)
    rows = [fill, 8191, 8192, 8193, fill + n - 1]
    got = out.float().cpu().double().numpy()
    for i, want in zip(rows, _oracle_rows(q, k, v, rows)):
        d = np.abs(got[i - fill] - want)
        assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (i, d.max(), d.mean())
    ctx.close()
    rctx.close()


def test_prefill_larger_ring(dev, dec_module):
    """R = 8320 (W + 128): chunks of 64 across the wrap; the outputs equal those of the
    8192-slot ring stepped one token at a time (ring size is not observable)."""
    cfg = vst.config_default(vst.DEC)
    cfg.ring_slots = 8320
    big = vst.Module(cfg)
    fill, n = 8250, 150
    q, k, v = _dec_seq(24, 0, fill + n)
    out, ctx = _prefill(big, dev, q, k, v, fill, n)
    ref, rctx = _steps(dec_module, dev, q, k, v, fill, n)
    assert torch.equal(out, ref)
    ctx.close()
    rctx.close()
    big.close()


def test_prefill_arguments(dev, dec_module):
    """n = 0 is a no-op; a negative n, positions past max_position or tensors shorter than n
    tokens are refused with nothing enqueued and the ctx unchanged."""
    ctx = _Ctx(dec_module, dev)
    q, k, v = _dec_seq(25, 0, 4)
    out = torch.empty((4, 32, 128), dtype=torch.bfloat16, device=dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    vst.dec_prefill(ctx.handle, qd, kd, vd, out, n=0)
    assert vst.ctx_info_get(ctx.handle).abs_next == 0
    with pytest.raises(RuntimeError):
        vst.dec_prefill(ctx.handle, qd, kd, vd, out, n=-1)
    # past max_position: refused by the library (raw pointers bypass the binding's size check)
    with pytest.raises(RuntimeError):
        vst.dec_prefill(ctx.handle, qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                        n=dec_module.cfg.max_position + 1)
    # more tokens than the tensors hold: refused by the binding before the call
    with pytest.raises(ValueError):
        vst.dec_prefill(ctx.handle, qd, kd, vd, out, n=5)
    assert vst.ctx_info_get(ctx.handle).abs_next == 0
    assert vst.ctx_check(ctx.handle) == vst.OK
    ctx.close()
