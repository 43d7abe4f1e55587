"""The figures bench.py reports, checked on the CPU.

- The algorithmic work that every roofline fraction divides by, counted here by brute force
  from the masks and the ring rules (the ring from the oracle's own bookkeeping), and the
  totals quoted for the workloads (4.97e11 FLOP for the 32-layer 4416-frame stream, 33.57 MB
  per decoder layer-step at a full window).
- The split of a timed region between the kernels of a step.
- The DRAM-traffic lookup, which must go blank when a kernel's sources change after its
  capture.
"""
import json
import os
import shutil
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402


def _bare(cls, **fields):
    """An instance of a bench workload class holding only the fields its counting methods
    read (the constructors allocate GPU memory)."""
    obj = object.__new__(cls)
    obj.__dict__.update(fields)
    return obj


def _visible_pairs(n, left, right=0):
    """(query i, key j) pairs of an n-frame clip with 0 <= i - j < left or 0 < j - i < right."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    d = i - j
    return int(np.count_nonzero(((d >= 0) & (d < left)) | ((-d > 0) & (-d < right))))


def test_encoder_attention_flops_by_brute_force():
    w = _bare(bench.EncWorkload, L=2, S=3, pre=[0, 96, 1000], frames=700)
    pairs = sum(_visible_pairs(p + 700, bench.ENC_W) for p in w.pre)
    assert w.attn_flops() == 4.0 * bench.ENC_D * bench.ENC_H * 2 * pairs


def test_headline_encoder_flops():
    w = _bare(bench.EncWorkload, L=32, S=1, pre=[0], frames=4416)
    assert w.attn_flops() == 4.0 * 64 * 20 * 32 * _visible_pairs(4416, 750)
    assert abs(w.attn_flops() - 4.97e11) < 0.005e11


def test_compaction_bytes_follow_the_oracle_ring():
    for frames, feed, pre in ((4416, 50, [0]), (3000, 512, [0, 96, 1440]), (2000, 7, [5, 0])):
        sched = bench.enc_feed_schedule(frames, feed)
        w = _bare(bench.EncWorkload, L=3, S=len(pre), pre=pre, sched=sched, frames=frames)
        n = 0
        for p in pre:
            ring = oracle.RingState()
            for chunk in ([p] if p else []) + [c for (_, c) in sched]:
                ring.feed(chunk)
            n += ring.n_compactions
        per = 2 * 2 * bench.ENC_H * bench.ENC_W * bench.ENC_D * 2  # K and V, read and write
        assert w.compact_bytes() == n * 3 * per, (frames, feed, pre)
    # the headline stream: 4 compactions per layer
    w = _bare(bench.EncWorkload, L=1, S=1, pre=[0], sched=bench.enc_feed_schedule(4416, 50), frames=4416)
    assert w.compact_bytes() == 4 * 7_680_000


def test_decoder_bytes():
    w = _bare(bench.DecWorkload, L=1, steps=1)
    # a full 8192-key window: K and V of 8192 keys x 8 heads x 128 x 2 B, plus q, out, k, v
    assert w.kv_bytes([8192]) == 8192 * 8 * 128 * 2 * 2 + (32 * 128 * 2) * 2 + (8 * 128 * 2) * 2 == 33_574_912
    w = _bare(bench.DecWorkload, L=26, steps=3)
    keys = sum(min(p + t + 1, 8192) for p in (0, 100, 8190) for t in range(3))
    io = 3 * 3 * ((32 * 128 * 2) * 2 + (8 * 128 * 2) * 2)
    assert w.kv_bytes([0, 100, 8190]) == 26 * (keys * 8 * 128 * 2 * 2 + io)


def test_prefill_bytes_equal_one_token_steps():
    w = _bare(bench.PrefillWorkload, L=26, n=39)
    d = _bare(bench.DecWorkload, L=26, steps=39)
    assert w.kv_bytes() == d.kv_bytes([0])


def test_offline_flops_by_brute_force():
    for T, left, right in ((300, 16, 4), (300, 750, 0), (300, 750, 4), (257, 1, 1), (200, 1000, 1000)):
        w = _bare(bench.OfflineWorkload, T=T, B=3, left=left, right=right)
        assert w.flops_per_launch() == 4.0 * bench.ENC_D * bench.ENC_H * 3 * _visible_pairs(T, left, right), (T, left, right)


def test_region_split_between_kernels():
    prof = {"enc_attn_kernel": (10, 2.0), "compact_kernel": (5, 1.0), "dec_step_kernel": (0, 0.0)}
    # 6 ms of timed region, shared 2:1 by event time: 4 ms over 10 attention launches
    assert abs(bench.region_launch_us(prof, "enc_attn_kernel", 6.0) - 400.0) < 1e-9
    assert abs(bench.region_launch_us(prof, "compact_kernel", 6.0) - 400.0) < 1e-9


def test_traffic_lookup_goes_blank_when_sources_change(tmp_path, monkeypatch):
    csrc = tmp_path / "sliding_window_kv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in set(sum(bench.KERNEL_SOURCES.values(), ())):
        shutil.copy(os.path.join(ROOT, "sliding_window_kv_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha("dec_step_kernel")
    table = {"dec_step_kernel": {"dram_bytes_per_unit": 1.5, "source_sha": sha},
             "dec_step_kernel@dec_prefill39": {"dram_bytes_per_unit": 0.25, "source_sha": sha}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(table))
    assert bench.dram_traffic("dec_step_kernel", 1000.0) == 1500.0
    assert bench.dram_traffic("dec_step_kernel", 1000.0, "dec_prefill39") == 250.0   # its own launch shape
    assert bench.dram_traffic("dec_step_kernel", 1000.0, "dec_b64") == 1500.0        # falls back to the default
    assert bench.dram_traffic("dec_step_kernel", 1000.0, "dec_b64", fallback=False) is None
    assert bench.dram_traffic("compact_kernel", 1000.0) is None                      # never captured
    with open(csrc / "dec_step.cu", "a") as f:
        f.write("\n// edited after the capture\n")
    assert bench.dram_traffic("dec_step_kernel", 1000.0) is None
    assert bench.dram_traffic("dec_step_kernel", 1000.0, "dec_prefill39") is None
