"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element,
plus the bit-exact self-consistency the method promises (chunking and compaction schedules
are not observable; batched decode equals single-stream decode; ring size is not
observable). Tolerances: max|d| <= 2e-2 and mean|d| <= 2e-3 against the oracle on bf16
inputs with fp32 accumulation; bit-exact for ring bytes and for self-consistency.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_kv_gb300 import synth, vst

pytestmark = pytest.mark.gpu

MAX_TOL = 2e-2
MEAN_TOL = 2e-3


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


def _enc_inputs(seed, layer, T, H=20, D=64, device="cpu", first=0):
    q = synth.frames(synth.tensor_key(seed, layer, 0), first, T, H, D, device)
    k = synth.frames(synth.tensor_key(seed, layer, 1), first, T, H, D, device)
    v = synth.frames(synth.tensor_key(seed, layer, 2), first, T, H, D, device)
    return q, k, v


def _compare(gpu_out, want, tag=""):
    got = gpu_out.float().cpu().double().numpy().reshape(want.shape)
    d = np.abs(got - want)
    assert np.isfinite(got).all(), tag
    assert d.max() <= MAX_TOL, "%s max|d| %.3e" % (tag, d.max())
    assert d.mean() <= MEAN_TOL, "%s mean|d| %.3e" % (tag, d.mean())
    _report(tag or "whole output", [d])
    return d.max(), d.mean()


def _report(tag, ds):
    """Print the worst max|d| and the mean|d| over every sampled element (pytest -s shows it)."""
    if ds:
        allv = np.concatenate([x.ravel() for x in ds])
        print("parity %s: %d rows, max|d| %.3e, mean|d| %.3e" % (tag, len(ds), allv.max(), allv.mean()))


def _feed(module, q, k, v, chunks, compact_before=(), dev="cuda"):
    """Stream q/k/v through one fresh ctx in the given chunk sizes; returns out [T][H][D]."""
    ctx = vst.Ctx(module)
    T = q.shape[0]
    out = torch.empty_like(q, device=dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    t = 0
    for ci, n in enumerate(chunks):
        if ci in compact_before:
            vst.ctx_compact(ctx.handle)
        vst.enc_feed(ctx.handle, qd[t:t + n], kd[t:t + n], vd[t:t + n], out[t:t + n], n_new=n)
        t += n
    assert t == T
    torch.cuda.synchronize()
    assert vst.ctx_check(ctx.handle) == vst.OK
    info = ctx.info()
    ctx.close()
    return out, info


# ---------------------------------------------------------------- encoder

def test_enc_small_single_tile(dev, enc_module):
    q, k, v = _enc_inputs(101, 0, 60)
    out, _ = _feed(enc_module, q, k, v, [60])
    want = oracle.attention(synth.bits(q), synth.bits(k), synth.bits(v), window=750)
    _compare(out, want, "T=60")


def test_enc_config0_parity_and_bit_exact(dev, enc_module):
    """1 layer, 20 heads x 64, 1000 frames fed as 10 chunks of 100 with a compaction forced
    before chunk 9 (n_kv 800 -> 750): matches the oracle, and matches bit for bit a single
    1000-frame feed and the same chunking without the forced compaction."""
    q, k, v = _enc_inputs(1, 0, 1000)
    want = oracle.attention(synth.bits(q), synth.bits(k), synth.bits(v), window=750, threads=8)
    out_c, info = _feed(enc_module, q, k, v, [100] * 10, compact_before=(8,))
    assert (info.n_compactions, info.abs_base, info.n_kv) == (1, 50, 950)
    _compare(out_c, want, "chunks of 100 + compaction")
    out_1, info1 = _feed(enc_module, q, k, v, [1000])
    assert info1.n_compactions == 0
    out_n, _ = _feed(enc_module, q, k, v, [100] * 10)
    assert torch.equal(out_c, out_1)
    assert torch.equal(out_c, out_n)


@pytest.mark.parametrize("sched", ["ones_then_big", "ragged", "max_batch_edges", "empty_feeds"])
def test_enc_chunking_not_observable(dev, enc_module, sched):
    T = 1700
    q, k, v = _enc_inputs(7, 3, T)
    ref, _ = _feed(enc_module, q, k, v, [T])
    if sched == "ones_then_big":
        chunks = [1] * 37 + [T - 37]
    elif sched == "ragged":
        rng = np.random.default_rng(3)
        chunks = []
        while sum(chunks) < T:
            chunks.append(int(min(T - sum(chunks), rng.choice([1, 3, 49, 50, 127, 128, 129, 300, 511]))))
    elif sched == "max_batch_edges":
        chunks = [511, 512, 513, T - 1536]
    else:  # feeds of zero rows between 50-frame feeds change nothing
        chunks = []
        while sum(chunks) < T:
            chunks += [min(50, T - sum(chunks)), 0] + ([0] if len(chunks) % 7 == 0 else [])
    out, info = _feed(enc_module, q, k, v, chunks)
    assert info.abs_next == T
    assert torch.equal(out, ref), sched


@pytest.mark.parametrize("chunk_ms", [500, 1000, 2000, 20000])
def test_enc_chunk_sizes_of_the_pages(dev, enc_module, chunk_ms):
    """The streaming chunk sizes the family doc validates ("Voxtral Realtime", Capability
    Validation, Streaming row, item (3): 500, 1000, 2000 and 20000 ms) are feeds of 25, 50,
    100 and 1000 encoder frames at 50 frames per second. Over 2600 frames (compactions at
    every size) each gives the bits of one single feed."""
    T = 2600
    q, k, v = _enc_inputs(9, 0, T)
    ref, _ = _feed(enc_module, q, k, v, [T])
    n = chunk_ms // 20
    chunks = [min(n, T - a) for a in range(0, T, n)]
    out, info = _feed(enc_module, q, k, v, chunks)
    assert info.abs_next == T and info.n_compactions >= 1
    assert torch.equal(out, ref), chunk_ms


def test_enc_long_stream_parity_sampled(dev, enc_module):
    """5000 frames in 50-frame feeds (lazy compactions): sampled rows against the oracle
    computed from each row's own window."""
    T = 5000
    q, k, v = _enc_inputs(2, 5, T)
    out, info = _feed(enc_module, q, k, v, [50] * 100)
    st = oracle.RingState()
    for _ in range(100):
        st.feed(50)
    assert (info.n_kv, info.abs_base, info.n_compactions) == (st.n_kv, st.abs_base, st.n_compactions)
    qb, kb, vb = synth.bits(q), synth.bits(k), synth.bits(v)
    rows = [0, 1, 749, 750, 1499, 1500, 1536, 2287, 3333, 4999]
    got = out.float().cpu().double().numpy()
    ds = []
    for i in rows:
        j0 = max(0, i - 749)
        want = oracle.attention_row(qb[i], kb[j0:i + 1], vb[j0:i + 1], i, 750)
        d = np.abs(got[i] - want)
        ds.append(d)
        assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (i, d.max(), d.mean())
    _report("5000 frames in 50-frame feeds", ds)


class TorchCtx:
    """A ctx on caller-provided memory (a torch uint8 buffer), so the rings can be viewed."""

    def __init__(self, module, dev):
        cfg = module.cfg
        self.mem = torch.zeros(vst.ctx_bytes(module.handle), dtype=torch.uint8, device=dev)
        self.handle = vst.ctx_create(module.handle, self.mem.data_ptr(), self.mem.numel())
        info = vst.ctx_info_get(self.handle)
        n = cfg.n_kv_heads * cfg.ring_slots * cfg.head_dim * 2
        shape = (cfg.n_kv_heads, cfg.ring_slots, cfg.head_dim)
        ko = info.k_ring - self.mem.data_ptr()
        vo = info.v_ring - self.mem.data_ptr()
        self.k_ring = self.mem[ko:ko + n].view(torch.bfloat16).view(shape)
        self.v_ring = self.mem[vo:vo + n].view(torch.bfloat16).view(shape)

    def info(self):
        return vst.ctx_info_get(self.handle)

    def close(self):
        vst.ctx_destroy(self.handle)


def test_enc_ring_after_compaction_bit_exact(dev, enc_module):
    """After compaction slot s holds what slot n_kv - 750 + s held before (bit for bit), and
    the appended keys are the oracle's rotated keys rounded to bf16."""
    T = 1000
    q, k, v = _enc_inputs(11, 0, T)
    ctx = TorchCtx(enc_module, dev)
    out = torch.empty_like(q, device=dev)
    vst.enc_feed(ctx.handle, q.to(dev), k.to(dev), v.to(dev), out)
    torch.cuda.synchronize()
    before_k = ctx.k_ring.clone()
    before_v = ctx.v_ring.clone()
    vst.ctx_compact(ctx.handle)
    torch.cuda.synchronize()
    info = ctx.info()
    assert (info.n_kv, info.abs_base, info.n_compactions) == (750, 250, 1)
    assert torch.equal(ctx.k_ring[:, :750], before_k[:, 250:1000])
    assert torch.equal(ctx.v_ring[:, :750], before_v[:, 250:1000])
    # slot s now holds absolute frame 250 + s: rotated K (bf16) and V as fed
    krot = oracle.rope_rows(synth.bits(k), 0)
    got = ctx.k_ring[:, :750].float().cpu().double().numpy().transpose(1, 0, 2)
    want = krot[250:1000]
    assert np.abs(got - want).max() <= np.abs(want).max() * 2 ** -8 + 1e-6
    assert torch.equal(ctx.v_ring[:, :750].cpu(), v[250:1000].transpose(0, 1).contiguous())
    # the ring keeps serving: next frames attend across the compacted rows
    q2, k2, v2 = _enc_inputs(11, 0, 200, first=1000)
    out2 = torch.empty_like(q2, device=dev)
    vst.enc_feed(ctx.handle, q2.to(dev), k2.to(dev), v2.to(dev), out2)
    torch.cuda.synchronize()
    qa, ka, va = (torch.cat([a, b]) for a, b in ((q, q2), (k, k2), (v, v2)))
    want2 = oracle.attention(synth.bits(qa), synth.bits(ka), synth.bits(va), window=750, rows=(1000, 1200),
                             threads=8)
    _compare(out2, want2, "after compaction")
    ctx.close()


def test_enc_batch_compaction_ring_bytes(dev, enc_module):
    """A batched feed of several query tiles on which some contexts compact and some do not.
    Three contexts fed together: fill 1100 + 300 (the move overlaps itself and the batch
    lands inside the old source rows), fill 1530 + 300 (disjoint move, batch inside the old
    source rows) and fill 200 + 300 (no compaction). Ring bytes, ring state and outputs equal
    those of each context compacted explicitly and then fed alone, and rows match the
    oracle."""
    fills, b = [1100, 1530, 200], 300
    seqs = [_enc_inputs(13, s, fills[s] + b) for s in range(3)]

    def prefilled(s):
        ctx = TorchCtx(enc_module, dev)
        o = torch.empty((fills[s], 20, 64), dtype=torch.bfloat16, device=dev)
        vst.enc_feed(ctx.handle, *(x[:fills[s]].to(dev) for x in seqs[s]), o)
        return ctx

    fused = [prefilled(s) for s in range(3)]
    Q, K, V = (torch.stack([seqs[s][i][fills[s]:] for s in range(3)]).to(dev) for i in range(3))
    OUT = torch.empty_like(Q)
    vst.enc_feed_batch([c.handle for c in fused], Q, K, V, OUT, b)
    torch.cuda.synchronize()
    got = OUT.float().cpu().double().numpy()
    ds = []
    for s in range(3):
        ref = prefilled(s)
        if fills[s] + b > 1536:
            vst.ctx_compact(ref.handle)
        out = torch.empty((b, 20, 64), dtype=torch.bfloat16, device=dev)
        vst.enc_feed(ref.handle, *(x[fills[s]:].to(dev) for x in seqs[s]), out)
        torch.cuda.synchronize()
        assert vst.ctx_check(fused[s].handle) == vst.OK and vst.ctx_check(ref.handle) == vst.OK
        a, r = fused[s].info(), ref.info()
        assert (a.n_kv, a.abs_base, a.abs_next, a.n_compactions) == (r.n_kv, r.abs_base, r.abs_next, r.n_compactions)
        assert torch.equal(fused[s].k_ring, ref.k_ring), s
        assert torch.equal(fused[s].v_ring, ref.v_ring), s
        assert torch.equal(OUT[s], out), s
        qb, kb, vb = (synth.bits(x) for x in seqs[s])
        for i in (0, 127, 128, b - 1):
            p = fills[s] + i
            j0 = max(0, p - 749)
            want = oracle.attention_row(qb[p], kb[j0:p + 1], vb[j0:p + 1], p, 750)
            d = np.abs(got[s, i] - want)
            ds.append(d)
            assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (s, i, d.max(), d.mean())
        ref.close()
    _report("batched compaction rows", ds)
    for c in fused:
        c.close()


@pytest.mark.parametrize("n_ctx,step", [(4, 300), (8, 100)])
def test_enc_batch_equals_single(dev, enc_module, n_ctx, step):
    """Streams with staggered starts fed together through vst_enc_feed_batch give the same
    bits as each stream fed alone. With 8 contexts x 20 heads the batched launch runs one
    CTA per query tile while a lone 100-frame feed splits its key tiles across CTAs: the two
    launch shapes must agree bit for bit."""
    T = 900
    offsets = [0, 96, 192, 700, 13, 1536, 1537, 3000][:n_ctx]
    ins = [_enc_inputs(5, s, T) for s in range(n_ctx)]
    pres = [_enc_inputs(55, s, offsets[s]) if offsets[s] else None for s in range(n_ctx)]

    def prefeed(ctx, s):
        if pres[s] is not None:
            o = torch.empty_like(pres[s][0], device=dev)
            vst.enc_feed(ctx.handle, *(t.to(dev) for t in pres[s]), o)

    singles = []
    for s in range(n_ctx):
        ctx = vst.Ctx(enc_module)
        prefeed(ctx, s)
        out = torch.empty_like(ins[s][0], device=dev)
        for t0 in range(0, T, step):
            vst.enc_feed(ctx.handle, *(t[t0:t0 + step].to(dev) for t in ins[s]), out[t0:t0 + step])
        singles.append(out)
        ctx.close()
    ctxs = [vst.Ctx(enc_module) for _ in range(n_ctx)]
    for s in range(n_ctx):
        prefeed(ctxs[s], s)
    Q, K, V = (torch.stack([ins[s][i] for s in range(n_ctx)]).to(dev) for i in range(3))
    OUT = torch.empty_like(Q)
    for t0 in range(0, T, step):
        o = torch.empty_like(Q[:, t0:t0 + step].contiguous())
        vst.enc_feed_batch([c.handle for c in ctxs], Q[:, t0:t0 + step].contiguous(),
                           K[:, t0:t0 + step].contiguous(), V[:, t0:t0 + step].contiguous(), o, step)
        OUT[:, t0:t0 + step] = o
    torch.cuda.synchronize()
    for s in range(n_ctx):
        assert torch.equal(OUT[s], singles[s]), s
        assert ctxs[s].info().abs_next == offsets[s] + T
    for c in ctxs:
        c.close()


def test_enc_16_unstaggered_streams_512_batches(dev, enc_module):
    """16 streams that all start at position 0, fed four 512-frame batches together (the
    fourth after a compaction of all 16 rings in one launch): every loop-shape launch covers
    the same positions in every context, from one key tile per query tile at the start of
    the clip to seven after the compaction, with ring slots below zero for the first key
    tile. Sampled rows of three streams against the oracle; stream 0 re-fed alone in
    50-frame feeds (the split shape) gives the same bits."""
    S, T, B = 16, 2048, 512
    seqs = [_enc_inputs(7, s, T) for s in range(S)]
    ctxs = [vst.Ctx(enc_module) for _ in range(S)]
    Q, K, V = (torch.stack([seqs[s][i] for s in range(S)]).to(dev) for i in range(3))
    OUT = torch.empty_like(Q)
    for t0 in range(0, T, B):
        o = torch.empty_like(Q[:, t0:t0 + B].contiguous())
        vst.enc_feed_batch([c.handle for c in ctxs], Q[:, t0:t0 + B].contiguous(), K[:, t0:t0 + B].contiguous(),
                           V[:, t0:t0 + B].contiguous(), o, B)
        OUT[:, t0:t0 + B] = o
    torch.cuda.synchronize()
    for c in ctxs:
        assert vst.ctx_check(c.handle) == vst.OK
        info = c.info()
        assert (info.n_kv, info.abs_base, info.abs_next, info.n_compactions) == (1262, 786, 2048, 1)
    got = OUT.float().cpu().double().numpy()
    ds = []
    for s in (0, 7, 15):
        qb, kb, vb = (synth.bits(x) for x in seqs[s])
        for i in (0, 127, 128, 511, 512, 1535, 1536, 1663, 2047):
            j0 = max(0, i - 749)
            want = oracle.attention_row(qb[i], kb[j0:i + 1], vb[j0:i + 1], i, 750)
            d = np.abs(got[s, i] - want)
            ds.append(d)
            assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (s, i, d.max(), d.mean())
    _report("16 streams from position 0, 512-frame batches", ds)
    alone, _ = _feed(enc_module, *seqs[0], [50] * (T // 50) + [T % 50])
    assert torch.equal(alone, OUT[0])
    for c in ctxs:
        c.close()


def test_enc_16_streams_512_batches(dev, enc_module):
    """The 16-stream launch configuration: streams with staggered starts (a first feed of
    96 s frames), then 512-frame batches through vst_enc_feed_batch (every batch launch is
    the loop shape over 16 contexts x 20 heads x 4 query tiles, with a compaction before the
    third). Sampled rows against the oracle; one stream re-fed alone in 50-frame feeds (the
    split shape) gives the same bits as in the batch."""
    S, T, B = 16, 1536, 512
    offsets = [96 * s for s in range(S)]
    seqs = [_enc_inputs(9, s, offsets[s] + T) for s in range(S)]
    ctxs = [vst.Ctx(enc_module) for _ in range(S)]
    for s in range(S):
        if offsets[s]:
            o = torch.empty((offsets[s], 20, 64), dtype=torch.bfloat16, device=dev)
            vst.enc_feed(ctxs[s].handle, *(x[:offsets[s]].to(dev) for x in seqs[s]), o)
    Q, K, V = (torch.stack([seqs[s][i][offsets[s]:] for s in range(S)]).to(dev) for i in range(3))
    OUT = torch.empty_like(Q)
    for t0 in range(0, T, B):
        o = torch.empty_like(Q[:, t0:t0 + B].contiguous())
        vst.enc_feed_batch([c.handle for c in ctxs], Q[:, t0:t0 + B].contiguous(), K[:, t0:t0 + B].contiguous(),
                           V[:, t0:t0 + B].contiguous(), o, B)
        OUT[:, t0:t0 + B] = o
    torch.cuda.synchronize()
    for s in range(S):
        assert vst.ctx_check(ctxs[s].handle) == vst.OK
        assert ctxs[s].info().abs_next == offsets[s] + T
    got = OUT.float().cpu().double().numpy()
    ds = []
    for s in (0, 5, 15):
        qb, kb, vb = (synth.bits(x) for x in seqs[s])
        for i in (0, 1, 511, 512, 1023, 1024, 1535):
            p = offsets[s] + i
            j0 = max(0, p - 749)
            want = oracle.attention_row(qb[p], kb[j0:p + 1], vb[j0:p + 1], p, 750)
            d = np.abs(got[s, i] - want)
            ds.append(d)
            assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (s, i, d.max(), d.mean())
    _report("16 staggered streams, 512-frame batches", ds)
    s = 7
    alone, _ = _feed(enc_module, *seqs[s], [offsets[s]] + [50] * (T // 50) + [T % 50])
    assert torch.equal(alone[offsets[s]:], OUT[s])
    for c in ctxs:
        c.close()


# ---------------------------------------------------------------- decoder

def _dec_seq(seed, stream, layer, n_tok, device="cpu", first=0):
    q = synth.frames(synth.tensor_key(seed, stream, layer, 0), first, n_tok, 32, 128, device)
    k = synth.frames(synth.tensor_key(seed, stream, layer, 1), first, n_tok, 8, 128, device)
    v = synth.frames(synth.tensor_key(seed, stream, layer, 2), first, n_tok, 8, 128, device)
    return q, k, v


def _run_dec(module, q, k, v, fill, steps, dev="cuda", ring_cfg=None):
    """Append `fill` tokens, then run `steps` decoder steps; returns out [steps][32][128]."""
    m = module
    ctx = vst.Ctx(m)
    if fill:
        vst.dec_append(ctx.handle, k[:fill].to(dev), v[:fill].to(dev))
    outs = torch.empty((steps, 32, 128), dtype=torch.bfloat16, device=dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    for s in range(steps):
        t = fill + s
        vst.dec_step([ctx.handle], qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], outs[s:s + 1])
    torch.cuda.synchronize()
    assert vst.ctx_check(ctx.handle) == vst.OK
    ctx.close()
    return outs


def test_dec_short_parity(dev, dec_module):
    n = 300
    q, k, v = _dec_seq(3, 0, 0, n)
    outs = _run_dec(dec_module, q, k, v, fill=0, steps=n)
    want = oracle.attention(synth.bits(q), synth.bits(k), synth.bits(v), window=8192, threads=8)
    _compare(outs, want, "decoder from empty")


def test_dec_wrap_parity_and_ring_ab(dev, dec_module):
    """Fill past the 8192 window so the modulo ring wraps, then step across more wraps;
    compare sampled steps with the oracle and the whole run with a 16384-slot ring."""
    fill, steps = 8190, 40
    n = fill + steps
    q, k, v = _dec_seq(3, 1, 0, n)
    outs = _run_dec(dec_module, q, k, v, fill=fill, steps=steps)
    cfg = vst.config_default(vst.DEC)
    cfg.ring_slots = 16384
    big = vst.Module(cfg)
    outs_big = _run_dec(big, q, k, v, fill=fill, steps=steps)
    big.close()
    assert torch.equal(outs, outs_big)
    qb, kb, vb = synth.bits(q), synth.bits(k), synth.bits(v)
    got = outs.float().cpu().double().numpy()
    for s in (0, 1, 2, 17, 39):
        i = fill + s
        j0 = max(0, i - 8191)
        want = oracle.attention_row(qb[i], kb[j0:i + 1], vb[j0:i + 1], i, 8192)
        d = np.abs(got[s] - want)
        assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (s, d.max(), d.mean())


def test_dec_batched_equals_single(dev, dec_module):
    """One vst_dec_step over 6 contexts with different fills = 6 single-stream steps."""
    fills = [0, 1, 127, 128, 4000, 9000]
    steps = 3
    seqs = [_dec_seq(4, s, 0, f + steps) for s, f in enumerate(fills)]
    singles = [_run_dec(dec_module, *seqs[s], fill=f, steps=steps) for s, f in enumerate(fills)]
    ctxs = [vst.Ctx(dec_module) for _ in fills]
    for c, (q, k, v), f in zip(ctxs, seqs, fills):
        if f:
            vst.dec_append(c.handle, k[:f].to(dev), v[:f].to(dev))
    for s in range(steps):
        Q = torch.stack([q[f + s] for (q, k, v), f in zip(seqs, fills)]).to(dev)
        K = torch.stack([k[f + s] for (q, k, v), f in zip(seqs, fills)]).to(dev)
        V = torch.stack([v[f + s] for (q, k, v), f in zip(seqs, fills)]).to(dev)
        O = torch.empty_like(Q)
        vst.dec_step([c.handle for c in ctxs], Q, K, V, O)
        for i in range(len(fills)):
            assert torch.equal(O[i], singles[i][s]), (i, s)
    for c in ctxs:
        c.close()


def test_dec_64_streams_uniform_fill_sampled(dev, dec_module):
    """The 64-stream decoder workload in the launch configuration the benchmark times: one
    layer of 64 contexts whose caches are filled to lengths drawn uniformly from [1, 8192]
    (seed 4, the same recipe: 81 to 8132 keys), then 4 batched steps. The shortest, the
    median and the longest stream are compared with the oracle, on each row's own window,
    at the first and the last step."""
    seed, S, steps, W = 4, 64, 4, 8192
    fills = synth.uniform_int(synth.tensor_key(seed, 99), S, 1, W)
    ctxs = [vst.Ctx(dec_module) for _ in range(S)]
    qs, ks, vs = [], [], []
    for s, f in enumerate(fills):
        k = synth.frames(synth.tensor_key(seed, s, 0, 1), 0, f + steps, 8, 128, dev)
        v = synth.frames(synth.tensor_key(seed, s, 0, 2), 0, f + steps, 8, 128, dev)
        vst.dec_append(ctxs[s].handle, k[:f], v[:f])
        qs.append(synth.frames(synth.tensor_key(seed, s, 0, 0), f, steps, 32, 128, dev))
        ks.append(k[f:])
        vs.append(v[f:])
    Q, K, V = (torch.stack(x, 1).contiguous() for x in (qs, ks, vs))  # [steps][S][...]
    O = torch.empty_like(Q)
    for t in range(steps):
        vst.dec_step([c.handle for c in ctxs], Q[t], K[t], V[t], O[t])
    torch.cuda.synchronize()
    for c in ctxs:
        assert vst.ctx_check(c.handle) == vst.OK
        c.close()
    got = O.float().cpu().double().numpy()
    order = sorted(range(S), key=lambda s: fills[s])
    for s in (order[0], order[S // 2], order[-1]):
        f = fills[s]
        qb = synth.bits(synth.frames(synth.tensor_key(seed, s, 0, 0), f, steps, 32, 128, "cpu"))
        for t in (0, steps - 1):
            i = f + t
            j0 = max(0, i - W + 1)
            kb = synth.bits(synth.frames(synth.tensor_key(seed, s, 0, 1), j0, i - j0 + 1, 8, 128, "cpu"))
            vb = synth.bits(synth.frames(synth.tensor_key(seed, s, 0, 2), j0, i - j0 + 1, 8, 128, "cpu"))
            want = oracle.attention_row(qb[t], kb, vb, i, W)
            d = np.abs(got[t, s] - want)
            assert np.isfinite(got[t, s]).all(), (s, t)
            assert d.max() <= MAX_TOL and d.mean() <= MEAN_TOL, (s, f, t, d.max(), d.mean())


def test_dec_batch_over_64_streams(dev, dec_module):
    """70 streams in one vst_dec_step call: the library launches them as 64 + 6 jobs. Every
    stream's rows equal the single-stream step's, fills from empty to past one tile."""
    n, steps = 70, 2
    fills = [(37 * s) % 300 for s in range(n)]
    seqs = [_dec_seq(14, s, 0, f + steps) for s, f in enumerate(fills)]
    ctxs = [vst.Ctx(dec_module) for _ in range(n)]
    for c, (q, k, v), f in zip(ctxs, seqs, fills):
        if f:
            vst.dec_append(c.handle, k[:f].to(dev), v[:f].to(dev))
    outs = []
    for s in range(steps):
        Q, K, V = (torch.stack([seqs[j][i][fills[j] + s] for j in range(n)]).to(dev) for i in range(3))
        O = torch.empty_like(Q)
        vst.dec_step([c.handle for c in ctxs], Q, K, V, O)
        outs.append(O)
    torch.cuda.synchronize()
    for c in ctxs:
        assert vst.ctx_check(c.handle) == vst.OK
        c.close()
    for i in (0, 1, 63, 64, 69):
        single = _run_dec(dec_module, *seqs[i], fill=fills[i], steps=steps)
        for s in range(steps):
            assert torch.equal(outs[s][i], single[s]), (i, s)


def test_enc_batch_over_64_contexts(dev, enc_module):
    """66 encoder contexts in one vst_enc_feed_batch call: launched as 64 contexts (the loop
    shape) and 2 (the split shape for a one-tile batch), with compactions due in both groups.
    Every context's rows equal those of the context fed alone."""
    n, T, step = 66, 1600, 100
    pre = [1400 + (s % 3) * 40 for s in range(n)]     # every context compacts during the feeds
    seqs = [_enc_inputs(15, s, pre[s] + T) for s in range(n)]

    def prefed(s):
        ctx = vst.Ctx(enc_module)
        o = torch.empty((pre[s], 20, 64), dtype=torch.bfloat16, device=dev)
        vst.enc_feed(ctx.handle, *(x[:pre[s]].to(dev) for x in seqs[s]), o)
        return ctx

    ctxs = [prefed(s) for s in range(n)]
    Q, K, V = (torch.stack([seqs[s][i][pre[s]:] for s in range(n)]).to(dev) for i in range(3))
    OUT = torch.empty_like(Q)
    for t0 in range(0, T, step):
        o = torch.empty_like(Q[:, t0:t0 + step].contiguous())
        vst.enc_feed_batch([c.handle for c in ctxs], Q[:, t0:t0 + step].contiguous(),
                           K[:, t0:t0 + step].contiguous(), V[:, t0:t0 + step].contiguous(), o, step)
        OUT[:, t0:t0 + step] = o
    torch.cuda.synchronize()
    for c in ctxs:
        assert vst.ctx_check(c.handle) == vst.OK
        assert c.info().n_compactions >= 1
        c.close()
    for s in (0, 1, 63, 64, 65):
        ctx = prefed(s)
        out = torch.empty((T, 20, 64), dtype=torch.bfloat16, device=dev)
        for t0 in range(0, T, step):
            vst.enc_feed(ctx.handle, *(x[pre[s] + t0:pre[s] + t0 + step].to(dev) for x in seqs[s]),
                         out[t0:t0 + step])
        torch.cuda.synchronize()
        ctx.close()
        assert torch.equal(OUT[s], out), s


def test_dec_append_ring_contents(dev, dec_module):
    """Token p lands in slot p % 8192 as bf16(RoPE(k, p)) (within bf16 rounding of the fp64
    oracle) and V bit for bit; the step path writes the same bytes as the append path."""
    n = 8192 + 300
    _, k, v = _dec_seq(9, 0, 0, n)
    ctx = TorchCtx(dec_module, dev)
    vst.dec_append(ctx.handle, k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    pos = np.arange(n - 8192, n)
    slots = torch.from_numpy(pos % 8192).to(dev)
    krot = oracle.rope_rows(synth.bits(k[n - 8192:]), n - 8192)
    got = ctx.k_ring[:, slots].float().cpu().double().numpy().transpose(1, 0, 2)
    assert np.abs(got - krot).max() <= np.abs(krot).max() * 2 ** -8 + 1e-6
    assert torch.equal(ctx.v_ring[:, slots].cpu(), v[n - 8192:].transpose(0, 1).contiguous())
    # one more token through the step path: same bytes as appending it
    q1, k1, v1 = _dec_seq(9, 0, 0, 1, first=n)
    ctx2 = TorchCtx(dec_module, dev)
    vst.dec_append(ctx2.handle, torch.cat([k, k1]).to(dev), torch.cat([v, v1]).to(dev))
    o = torch.empty((1, 32, 128), dtype=torch.bfloat16, device=dev)
    vst.dec_step([ctx.handle], q1.to(dev), k1.to(dev), v1.to(dev), o)
    torch.cuda.synchronize()
    assert torch.equal(ctx.k_ring, ctx2.k_ring)
    assert torch.equal(ctx.v_ring, ctx2.v_ring)
    ctx.close()
    ctx2.close()


def test_interleaved_contexts_bit_exact(dev, enc_module, dec_module):
    """Layers of a stream are different contexts called one after another on one CUDA
    stream; a launch may then fetch its ring tiles while the previous kernel (another
    context) is still running, and a compaction may copy its ring beside that kernel's tail.
    Feeding three encoder contexts and three decoder contexts round-robin must give the same
    bits as running each context alone."""
    # encoder: 3 contexts, 2024 frames each: 50-frame feeds, one 300-frame feed, then 512- and
    # 50-frame feeds, so that every context compacts right after another context's attention
    sched = [50] * 6 + [300] + [50] * 6 + [512, 50, 512, 50]
    ins = [_enc_inputs(31, l, sum(sched)) for l in range(3)]
    alone = [_feed(enc_module, *ins[l], sched)[0] for l in range(3)]
    ctxs = [vst.Ctx(enc_module) for _ in range(3)]
    outs = [torch.empty_like(ins[l][0], device=dev) for l in range(3)]
    dins = [[t.to(dev) for t in ins[l]] for l in range(3)]
    t = 0
    for n in sched:
        for l in range(3):
            q, k, v = dins[l]
            vst.enc_feed(ctxs[l].handle, q[t:t + n], k[t:t + n], v[t:t + n], outs[l][t:t + n])
        t += n
    torch.cuda.synchronize()
    for l in range(3):
        assert vst.ctx_info_get(ctxs[l].handle).n_compactions >= 1
        assert torch.equal(outs[l], alone[l]), l
        ctxs[l].close()
    # decoder: 3 contexts with different fills, 6 steps round-robin
    fills = [100, 8190, 9001]
    seqs = [_dec_seq(32, s, 0, f + 6) for s, f in enumerate(fills)]
    alone = [_run_dec(dec_module, *seqs[s], fill=f, steps=6) for s, f in enumerate(fills)]
    dctx = [vst.Ctx(dec_module) for _ in fills]
    for c, (q, k, v), f in zip(dctx, seqs, fills):
        vst.dec_append(c.handle, k[:f].to(dev), v[:f].to(dev))
    got = [torch.empty((6, 32, 128), dtype=torch.bfloat16, device=dev) for _ in fills]
    dseq = [[x.to(dev) for x in sq] for sq in seqs]
    for st in range(6):
        for s, f in enumerate(fills):
            q, k, v = dseq[s]
            vst.dec_step([dctx[s].handle], q[f + st:f + st + 1], k[f + st:f + st + 1], v[f + st:f + st + 1],
                         got[s][st:st + 1])
    torch.cuda.synchronize()
    for s in range(3):
        assert torch.equal(got[s], alone[s]), s
        dctx[s].close()


def test_all_paths_interleaved_bit_exact(dev, enc_module, dec_module):
    """Every kernel of the library is chained by programmatic dependent launch, so a launch
    may start while the previous one, on another context or another path, still runs.
    Streaming feeds (both launch shapes, with a compaction), decoder steps, prefill chunks
    and offline passes issued round-robin on one CUDA stream, with the offline plan reused
    from one pass to the next, must give the same bits as each run alone."""
    T = 1700
    q, k, v = _enc_inputs(61, 0, T)
    enc_alone = _feed(enc_module, q, k, v, [512, 50, 512, 50, 512, 64])[0]
    off_in = [_enc_inputs(62 + i, 0, 600) for i in range(3)]
    plan = vst.Offline(enc_module, 1, 600)
    off_alone = []
    for i in range(3):
        o = torch.empty((1, 600, 20, 64), dtype=torch.bfloat16, device=dev)
        plan.run(*(x[None].to(dev) for x in off_in[i]), o, 750 if i != 1 else 16, 0 if i != 1 else 4)
        off_alone.append(o)
    fill = 8150
    dq, dk, dv = _dec_seq(63, 0, 0, fill + 100)
    dec_alone = _run_dec(dec_module, dq, dk, dv, fill=fill, steps=100)
    torch.cuda.synchronize()

    ectx = vst.Ctx(enc_module)
    dctx = vst.Ctx(dec_module)
    vst.dec_append(dctx.handle, dk[:fill].to(dev), dv[:fill].to(dev))
    eq, ek, ev = q.to(dev), k.to(dev), v.to(dev)
    qd, kd, vd = dq.to(dev), dk.to(dev), dv.to(dev)
    enc_out = torch.empty_like(eq)
    dec_out = torch.empty((100, 32, 128), dtype=torch.bfloat16, device=dev)
    off_out = [torch.empty((1, 600, 20, 64), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    t = 0
    dsteps = [("step", 1), ("prefill", 39), ("step", 1), ("prefill", 59)]
    d = 0
    for i, n in enumerate([512, 50, 512, 50, 512, 64]):
        vst.enc_feed(ectx.handle, eq[t:t + n], ek[t:t + n], ev[t:t + n], enc_out[t:t + n])
        t += n
        if i < len(dsteps):
            kind, m = dsteps[i]
            a = fill + d
            if kind == "step":
                vst.dec_step([dctx.handle], qd[a:a + 1], kd[a:a + 1], vd[a:a + 1], dec_out[d:d + 1])
            else:
                vst.dec_prefill(dctx.handle, qd[a:a + m], kd[a:a + m], vd[a:a + m], dec_out[d:d + m])
            d += m
        if i < 3:
            plan.run(*(x[None].to(dev) for x in off_in[i]), off_out[i], 750 if i != 1 else 16, 0 if i != 1 else 4)
    torch.cuda.synchronize()
    assert vst.ctx_check(ectx.handle) == vst.OK and vst.ctx_check(dctx.handle) == vst.OK
    assert plan.check() == vst.OK
    assert torch.equal(enc_out, enc_alone)
    assert d == 100 and torch.equal(dec_out, dec_alone)
    for i in range(3):
        assert torch.equal(off_out[i], off_alone[i]), i
    ectx.close()
    dctx.close()
    plan.close()
