"""vst_dec_step_noalloc: the decoder step for callers that cannot allocate device memory at
call time (a real-time streaming thread that must not block on cudaMalloc, or a process
whose device memory belongs to another allocator). Its scratch lives in a static device
array inside libvst; the test checks, through the C ABI, that two calls in a row give what
vst_dec_step gives on identical contexts, that those rows also agree with the fp64 oracle,
and that calls beyond the array's limit are refused. This file is collected last on purpose."""
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
    return torch.device("cuda:0")


def _make_streams(module, fills, seed, dev):
    ctxs = [vst.Ctx(module) for _ in fills]
    seqs = []
    for s, (c, f) in enumerate(zip(ctxs, fills)):
        q, k, v = (synth.frames(synth.tensor_key(seed, s, i), 0, f + 2, h, 128, dev)
                   for i, h in enumerate((32, 8, 8)))
        if f:
            vst.dec_append(c.handle, k[:f], v[:f])
        seqs.append((q, k, v))
    return ctxs, seqs


def test_noalloc_matches_dec_step_two_calls(dev):
    module = vst.Module(vst.DEC)
    fills = [0, 300, 8191, 9000]
    ref_ctxs, seqs = _make_streams(module, fills, 21, dev)
    na_ctxs, _ = _make_streams(module, fills, 21, dev)
    for step in range(2):  # two calls in a row share (and reuse) the static scratch
        Q = torch.stack([q[f + step] for (q, _, _), f in zip(seqs, fills)])
        K = torch.stack([k[f + step] for (_, k, _), f in zip(seqs, fills)])
        V = torch.stack([v[f + step] for (_, _, v), f in zip(seqs, fills)])
        ref = torch.empty_like(Q)
        got = torch.empty_like(Q)
        vst.dec_step([c.handle for c in ref_ctxs], Q, K, V, ref)
        vst.dec_step_noalloc([c.handle for c in na_ctxs], Q, K, V, got)
        torch.cuda.synchronize()
        d = (got.float() - ref.float()).abs()
        assert torch.isfinite(got.float()).all()
        assert d.max().item() <= MAX_TOL and d.mean().item() <= MEAN_TOL, (step, d.max().item())
        assert torch.equal(got, ref), step
        # each stream's row against the oracle computed from that row's own window
        outs = got.float().cpu().double().numpy()
        for s, ((q, k, v), f) in enumerate(zip(seqs, fills)):
            i = f + step
            j0 = max(0, i - 8191)
            qb, kb, vb = (synth.bits(x[:i + 1].cpu()) for x in (q, k, v))
            want = oracle.attention_row(qb[i], kb[j0:i + 1], vb[j0:i + 1], i, 8192)
            e = np.abs(outs[s] - want)
            assert e.max() <= MAX_TOL and e.mean() <= MEAN_TOL, (step, s, e.max(), e.mean())
    for c in ref_ctxs + na_ctxs:
        assert vst.ctx_check(c.handle) == vst.OK
        c.close()
    module.close()


def test_noalloc_rejects_more_streams_than_scratch(dev):
    module = vst.Module(vst.DEC)
    ctxs = [vst.Ctx(module) for _ in range(15)]  # 15 x 283 KB > 4 MiB
    q = torch.zeros((15, 32, 128), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((15, 8, 128), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    with pytest.raises(vst.VstError) as e:
        vst.dec_step_noalloc([c.handle for c in ctxs], q, kv, kv, out)
    assert e.value.status == vst.E_INVAL
    assert all(c.info().abs_next == 0 for c in ctxs)  # nothing enqueued, state unchanged
    for c in ctxs:
        c.close()
    module.close()
