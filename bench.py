#!/usr/bin/env python
"""Benchmark of the sliding-window KV attention path on one GB300.

Default line (the configuration the metric is quoted on): the encoder streaming workload
-- 32 layers x 20 heads x 64, window 750, ring 1536, one stream of 4416 frames fed in
50-frame chunks (88 x 50 + 16, four lazy compactions per layer). One step streams the whole
clip through all 32 layers (contexts reset at the start of the step), so every step covers
feed bookkeeping, compaction, RoPE + append and chunk attention. `value` is encoder frames
per second with inputs resident in HBM, measured on CUDA-graph replays of the step.

The same line carries every other configuration of the metric as an object: `dec`, the
decoder step workload (26 layers, GQA 32q/8kv x 128, KV filled to 8192, batch 1, 256 steps
across the ring wrap) in decoder steps per second, with its own end-to-end figure through
the C ABI; `dec_b64`, 64 decoder streams with fills uniform in [1, 8192]; `enc_long16`, 16
encoder streams with staggered starts in 512-frame batches (15300 frames each, many
compactions); and the next rows, `prefill` (the 39-token prompt) and `offline` (4 whole
clips). `--workload` runs one configuration alone (it prints the same kind of line).

Inputs are synthetic (seeded counter-based bf16 ~N(0,1), sliding_window_kv_gb300.synth);
the per-step inputs and caches exceed the 129 MB L2, so no flush is needed between steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "streamed enc frames/s + dec steps/s (1 GPU); % of HBM / BF16 tensor roofline"

ENC_H, ENC_D, ENC_W = 20, 64, 750
DEC_H, DEC_HK, DEC_D, DEC_W = 32, 8, 128, 8192

WORKLOADS = {
    # encoder streaming, 32 layers, one stream, 4416 frames in 50-frame feeds (default line)
    "enc_stream": dict(kind="enc", layers=32, frames=4416, feed=50, streams=1, seed=2, stagger=0),
    # encoder, one layer, 1000 frames in 100-frame feeds (small case)
    "enc_small": dict(kind="enc", layers=1, frames=1000, feed=100, streams=1, seed=1, stagger=0),
    # encoder, 16 concurrent streams, staggered starts (96*s frames), 512-frame batches
    "enc_long16": dict(kind="enc", layers=32, frames=15300, feed=512, streams=16, seed=5, stagger=96),
    # decoder, 26 layers, batch 1, KV filled to 8192
    "dec_b1": dict(kind="dec", layers=26, streams=1, fill="full", steps=256, seed=3),
    # decoder, 26 layers, 64 streams with fills uniform in [1, 8192]
    "dec_b64": dict(kind="dec", layers=26, streams=64, fill="uniform", steps=256, seed=4),
    # offline encoder, 32 layers, 4 whole clips of 4416 frames, the streaming mask (750, 0)
    "enc_offline4": dict(kind="offline", layers=32, clips=4, frames=4416, left=750, right=0, seed=8),
    # the same with a 4-frame right lookahead (the pages' (left, right) sliding mask)
    "enc_offline4_la": dict(kind="offline", layers=32, clips=4, frames=4416, left=750, right=4, seed=8),
    # decoder prefill, 26 layers, one stream: the 39-token prompt on an empty cache
    "dec_prefill39": dict(kind="prefill", layers=26, tokens=39, seed=6),
    # decoder prefill, 26 layers, one stream: a 512-token prompt on an empty cache
    "dec_prefill512": dict(kind="prefill", layers=26, tokens=512, seed=7),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="vst", choices=["vst", "reference"])
    ap.add_argument("--workload", default="enc_stream", choices=sorted(WORKLOADS))
    ap.add_argument("--no-dec", action="store_true",
                    help="skip the secondary objects of the default line (decoder, prefill, offline encoder)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dec-steps", type=int, default=256, help="decoder steps (decoder workloads and dec object)")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing

class Dist:
    def __init__(self, n_gpus: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if _cuda_ok() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if _cuda_ok() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def job_rate(self, units_per_rank: float, ms_local: float):
        """Whole-job throughput of the replicas: every rank processed `units_per_rank` units in
        its own `ms_local`, and the job took as long as the slowest rank. Returns (units per
        second over all ranks, the slowest rank's ms)."""
        ms = self.max(ms_local)
        return self.world * units_per_rank / (ms / 1e3), ms

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def want_cpu_baseline(args, dist) -> bool:
    """The oracle's CPU baseline is timed once, on a single-GPU run's only rank."""
    return not args.no_cpu and dist.world == 1 and dist.rank == 0


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a replica's inputs: each rank streams its own synthetic data (weak scaling)."""
    return seed + 1000 * rank


def _cuda_ok():
    import torch
    return torch.cuda.is_available()


# ---------------------------------------------------------------- clocks during timing

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int = 0):
        self.proc = None
        self.lines = []
        self.sel = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid:
                self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "100"] + self.sel, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def enc_feed_schedule(frames: int, feed: int):
    out, t = [], 0
    while t < frames:
        n = min(feed, frames - t)
        out.append((t, n))
        t += n
    return out


class EncWorkload:
    """Streams `frames` frames per stream through `layers` encoder layers in `feed`-frame
    chunks; stream s first gets an extra 96*s-frame feed (staggered start) when stagger.

    Inputs of one layer live in one contiguous buffer per tensor, laid out feed after feed
    as [S][n][H][D] blocks (what vst_enc_feed_batch takes), so a host copy of a layer's
    inputs is one copy per tensor."""

    def __init__(self, spec, dev, rank=0):
        import torch
        from sliding_window_kv_gb300 import synth, vst
        self.vst = vst
        self.spec = spec
        self.L, self.S = spec["layers"], spec["streams"]
        self.frames, self.feed = spec["frames"], spec["feed"]
        self.pre = [spec["stagger"] * s for s in range(self.S)]
        self.module = vst.Module(vst.ENC)
        self.ctxs = [[vst.Ctx(self.module) for _ in range(self.S)] for _ in range(self.L)]
        self.sched = enc_feed_schedule(self.frames, self.feed)
        seed = rank_seed(spec["seed"], rank)
        HD = ENC_H * ENC_D
        self.buf = []      # [layer][role] flat bf16 buffers (q, k, v, out)
        self.views = []    # [layer][role][feed] -> [S][n][H][D] views
        self.pbuf = []     # [layer][role] flat pre-feed buffers (all streams back to back)
        self.pviews = []   # [layer][role][stream] -> [pre_s][H][D]
        npre = sum(self.pre)
        for l in range(self.L):
            bl = [torch.empty(self.S * self.frames * HD, dtype=torch.bfloat16, device=dev) for _ in range(4)]
            pl = [torch.empty(max(1, npre) * HD, dtype=torch.bfloat16, device=dev) for _ in range(4)]
            vl = [[None] * len(self.sched) for _ in range(4)]
            pv = [[None] * self.S for _ in range(4)]
            for f, (t, n) in enumerate(self.sched):
                for i in range(4):
                    vl[i][f] = bl[i][self.S * t * HD:self.S * (t + n) * HD].view(self.S, n, ENC_H, ENC_D)
            off = 0
            for s in range(self.S):
                for i in range(4):
                    pv[i][s] = pl[i][off * HD:(off + self.pre[s]) * HD].view(self.pre[s], ENC_H, ENC_D)
                off += self.pre[s]
            for i in range(3):
                for s in range(self.S):
                    x = synth.frames(synth.tensor_key(seed, s, l, i), 0, self.pre[s] + self.frames, ENC_H, ENC_D, dev)
                    if self.pre[s]:
                        pv[i][s].copy_(x[:self.pre[s]])
                    for f, (t, n) in enumerate(self.sched):
                        vl[i][f][s].copy_(x[self.pre[s] + t:self.pre[s] + t + n])
                    del x
            self.buf.append(bl)
            self.pbuf.append(pl)
            self.views.append(vl)
            self.pviews.append(pv)
        self.frames_per_step = npre + self.S * self.frames
        self.in_bytes = self.L * 3 * (self.S * self.frames + npre) * HD * 2
        self.out_bytes = self.L * (self.S * self.frames + npre) * HD * 2

    def run_step(self, stream):
        vst = self.vst
        for l in range(self.L):
            for c in self.ctxs[l]:
                vst.ctx_reset(c.handle, stream)
        for l in range(self.L):
            pv = self.pviews[l]
            for s in range(self.S):
                if self.pre[s]:
                    vst.enc_feed(self.ctxs[l][s].handle, pv[0][s], pv[1][s], pv[2][s], pv[3][s], stream)
        for f, (t, n) in enumerate(self.sched):
            for l in range(self.L):
                q, k, v, o = (self.views[l][i][f] for i in range(4))
                if self.S == 1:
                    vst.enc_feed(self.ctxs[l][0].handle, q[0], k[0], v[0], o[0], stream, n_new=n)
                else:
                    vst.enc_feed_batch([c.handle for c in self.ctxs[l]], q, k, v, o, n, stream)

    def e2e_setup(self, stream):
        """End-to-end step as a streaming client runs it: the inputs of each feed (every
        layer's q, k, v) sit in one pinned host block and go to the GPU in one copy on a copy
        stream, the feed's C-ABI calls wait for that copy only, and the feed's outputs come
        back in one copy on a third stream. Device buffers are laid out feed-major to match."""
        import ctypes
        import torch
        vst = self.vst
        L = vst.lib()
        sp = vst._stream(stream)
        HD = ENC_H * ENC_D
        dev = self.buf[0][0].device
        feeds = []  # (rows per stream of this feed, offsets into each stream's input, is_pre)
        if sum(self.pre):
            feeds.append(("pre", None))
        for f, (t, n) in enumerate(self.sched):
            feeds.append(("feed", f))
        st = {"hin": [], "din": [], "hout": [], "dout": [], "calls": [], "arrays": []}
        resets = [(L.vst_ctx_reset, (c.handle, sp)) for l in range(self.L) for c in self.ctxs[l]]
        for kind, f in feeds:
            if kind == "pre":
                rows = sum(self.pre)
                src = [[self.pbuf[l][i][:rows * HD] for i in range(3)] for l in range(self.L)]
            else:
                t, n = self.sched[f]
                rows = self.S * n
                src = [[self.views[l][i][f].reshape(-1) for i in range(3)] for l in range(self.L)]
            per = rows * HD
            hin = torch.empty(self.L * 3 * per, dtype=torch.bfloat16, pin_memory=True)
            for l in range(self.L):
                for i in range(3):
                    hin[(l * 3 + i) * per:(l * 3 + i + 1) * per].copy_(src[l][i].cpu())
            din = torch.empty_like(hin, device=dev)
            hout = torch.empty(self.L * per, dtype=torch.bfloat16, pin_memory=True)
            dout = torch.empty_like(hout, device=dev)
            calls = []
            for l in range(self.L):
                q, k, v = (din[(l * 3 + i) * per:(l * 3 + i + 1) * per] for i in range(3))
                o = dout[l * per:(l + 1) * per]
                if kind == "pre":
                    off = 0
                    for s in range(self.S):
                        if self.pre[s]:
                            a = off * HD
                            calls.append((L.vst_enc_feed, (self.ctxs[l][s].handle, q[a:].data_ptr(), k[a:].data_ptr(),
                                                           v[a:].data_ptr(), self.pre[s], o[a:].data_ptr(), sp)))
                        off += self.pre[s]
                elif self.S == 1:
                    calls.append((L.vst_enc_feed, (self.ctxs[l][0].handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                   n, o.data_ptr(), sp)))
                else:
                    arr = (ctypes.c_void_p * self.S)(*[c.handle for c in self.ctxs[l]])
                    st["arrays"].append(arr)
                    calls.append((L.vst_enc_feed_batch, (arr, self.S, q.data_ptr(), k.data_ptr(), v.data_ptr(), n,
                                                         o.data_ptr(), sp)))
            st["hin"].append(hin)
            st["din"].append(din)
            st["hout"].append(hout)
            st["dout"].append(dout)
            st["calls"].append(calls)
        st["resets"] = resets
        st["copy"] = torch.cuda.Stream(dev)
        st["back"] = torch.cuda.Stream(dev)
        st["ev_in"] = [torch.cuda.Event() for _ in feeds]
        st["ev_out"] = [torch.cuda.Event() for _ in feeds]
        st["h2d"] = sum(x.numel() * 2 for x in st["hin"])
        st["d2h"] = sum(x.numel() * 2 for x in st["hout"])
        return st

    E2E_GROUP = 8  # feeds per cross-stream synchronisation

    def e2e_run(self, st, stream):
        """One end-to-end step, after everything already issued on `stream` (so a step's
        copies never overwrite inputs the previous step still reads). Every feed's inputs go
        in one copy and its outputs come back in one copy; the compute stream waits for the
        inputs, and the copy-back stream for the outputs, once per group of E2E_GROUP feeds
        (an event wait or record between two launches keeps them from overlapping, and the
        input copies run far ahead of the compute)."""
        import torch
        n = len(st["calls"])
        groups = [range(g, min(n, g + self.E2E_GROUP)) for g in range(0, n, self.E2E_GROUP)]
        st["copy"].wait_stream(stream)
        with torch.cuda.stream(st["copy"]):
            for gi, grp in enumerate(groups):
                for f in grp:
                    st["din"][f].copy_(st["hin"][f], non_blocking=True)
                st["ev_in"][gi].record(st["copy"])
        for fn, args in st["resets"]:
            if fn(*args) != 0:
                raise RuntimeError("vst_ctx_reset failed")
        for gi, grp in enumerate(groups):
            stream.wait_event(st["ev_in"][gi])
            for f in grp:
                for fn, args in st["calls"][f]:
                    if fn(*args) != 0:
                        raise RuntimeError("%s failed" % fn.__name__)
            st["ev_out"][gi].record(stream)
        with torch.cuda.stream(st["back"]):
            for gi, grp in enumerate(groups):
                st["back"].wait_event(st["ev_out"][gi])
                for f in grp:
                    st["hout"][f].copy_(st["dout"][f], non_blocking=True)
        stream.wait_stream(st["back"])

    def attn_flops(self):
        """Algorithmic FLOPs of kernel (b) per step: 4*D per visible (query, key) pair, per
        head and layer: sum over rows at absolute position p of min(W, p+1)."""
        pairs = 0
        for s in range(self.S):
            n = self.pre[s] + self.frames
            pairs += ENC_W * (ENC_W + 1) // 2 if n >= ENC_W else n * (n + 1) // 2
            pairs += max(0, n - ENC_W) * ENC_W
        return 4.0 * ENC_D * ENC_H * self.L * pairs

    def compact_bytes(self):
        """Algorithmic bytes of kernel (d) per step: each compaction reads and writes 750
        rows of K and V for every head (ring rule: compact before a batch that would not
        fit in 1536 rows; feeds pushed in batches of at most 512)."""
        n = 0
        for s in range(self.S):
            n_kv = 0
            for chunk in ([self.pre[s]] if self.pre[s] else []) + [c for (_, c) in self.sched]:
                t = chunk
                while t > 0:
                    b = min(512, t)
                    if n_kv + b > 1536:
                        n_kv = 750
                        n += 1
                    n_kv += b
                    t -= b
        return n * self.L * 2 * 2 * ENC_H * ENC_W * ENC_D * 2

    def close(self):
        for row in self.ctxs:
            for c in row:
                c.close()
        self.module.close()


def host_enqueue_cost(calls, burst=256):
    """Host time of a list of prepared C-ABI calls (fn, args), issued in bursts of `burst`
    calls after a synchronisation so that no call waits for room in the launch queue:
    (total ms, µs per call)."""
    import torch
    total = 0.0
    for i in range(0, len(calls), burst):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for fn, args in calls[i:i + burst]:
            if fn(*args) != 0:
                raise RuntimeError("%s failed" % fn.__name__)
        total += time.perf_counter() - t0
    torch.cuda.synchronize()
    return 1e3 * total, 1e6 * total / max(1, len(calls))


class DecWorkload:
    """26 decoder layers; each stream's cache filled (untimed) then `steps` decoder steps.
    Inputs of step t, layer l are [S][H][D] / [S][Hk][D] slices of per-layer buffers."""

    def __init__(self, spec, dev, n_steps, rank=0):
        import torch
        from sliding_window_kv_gb300 import synth, vst
        self.vst = vst
        self.L, self.S, self.steps = spec["layers"], spec["streams"], n_steps
        seed = rank_seed(spec["seed"], rank)
        if spec["fill"] == "full":
            self.fills = [DEC_W] * self.S
        else:
            self.fills = synth.uniform_int(synth.tensor_key(seed, 99), self.S, 1, DEC_W)
        self.module = vst.Module(vst.DEC)
        self.ctxs = [[vst.Ctx(self.module) for _ in range(self.S)] for _ in range(self.L)]
        self.Q, self.K, self.V, self.O = [], [], [], []
        for l in range(self.L):
            qs, ks, vs = [], [], []
            for s in range(self.S):
                f = self.fills[s]
                k = synth.frames(synth.tensor_key(seed, s, l, 1), 0, f + self.steps, DEC_HK, DEC_D, dev)
                v = synth.frames(synth.tensor_key(seed, s, l, 2), 0, f + self.steps, DEC_HK, DEC_D, dev)
                vst.dec_append(self.ctxs[l][s].handle, k[:f], v[:f])
                qs.append(synth.frames(synth.tensor_key(seed, s, l, 0), f, self.steps, DEC_H, DEC_D, dev))
                ks.append(k[f:])
                vs.append(v[f:])
            # [steps][S][...] so that step t is one contiguous [S][...] block
            self.Q.append(torch.stack(qs, 1).contiguous())
            self.K.append(torch.stack(ks, 1).contiguous())
            self.V.append(torch.stack(vs, 1).contiguous())
            self.O.append(torch.empty_like(self.Q[-1]))
            torch.cuda.synchronize()

    def positions(self):
        return [self.vst.ctx_info_get(self.ctxs[0][s].handle).abs_next for s in range(self.S)]

    def run_steps(self, stream):
        vst = self.vst
        for t in range(self.steps):
            for l in range(self.L):
                vst.dec_step([c.handle for c in self.ctxs[l]], self.Q[l][t], self.K[l][t], self.V[l][t],
                             self.O[l][t], stream)

    def e2e_setup(self, stream):
        """End-to-end decoding as a client runs it: each step's inputs (every layer's q, k, v
        for every stream) sit in one pinned host block and go to the GPU in one copy on a copy
        stream; the step's 26 vst_dec_step calls wait for that copy only, and the step's
        outputs come back in one copy on a third stream."""
        import ctypes
        import torch
        vst = self.vst
        L = vst.lib()
        sp = vst._stream(stream)
        dev = self.Q[0].device
        nq, nk = self.S * DEC_H * DEC_D, self.S * DEC_HK * DEC_D
        per_layer = nq + 2 * nk
        st = {"hin": [], "din": [], "hout": [], "dout": [], "calls": []}
        st["arrays"] = [(ctypes.c_void_p * self.S)(*[c.handle for c in self.ctxs[l]]) for l in range(self.L)]
        for t in range(self.steps):
            hin = torch.empty(self.L * per_layer, dtype=torch.bfloat16, pin_memory=True)
            for l in range(self.L):
                base = l * per_layer
                hin[base:base + nq].copy_(self.Q[l][t].reshape(-1).cpu())
                hin[base + nq:base + nq + nk].copy_(self.K[l][t].reshape(-1).cpu())
                hin[base + nq + nk:base + per_layer].copy_(self.V[l][t].reshape(-1).cpu())
            din = torch.empty_like(hin, device=dev)
            hout = torch.empty(self.L * nq, dtype=torch.bfloat16, pin_memory=True)
            dout = torch.empty_like(hout, device=dev)
            calls = []
            for l in range(self.L):
                base = l * per_layer
                calls.append((L.vst_dec_step, (st["arrays"][l], self.S, din[base:].data_ptr(),
                                               din[base + nq:].data_ptr(), din[base + nq + nk:].data_ptr(),
                                               dout[l * nq:].data_ptr(), sp)))
            st["hin"].append(hin)
            st["din"].append(din)
            st["hout"].append(hout)
            st["dout"].append(dout)
            st["calls"].append(calls)
        st["copy"] = torch.cuda.Stream(dev)
        st["back"] = torch.cuda.Stream(dev)
        n_groups = -(-self.steps // self.E2E_GROUP)
        st["ev_in"] = [torch.cuda.Event() for _ in range(n_groups)]
        st["ev_out"] = [torch.cuda.Event() for _ in range(n_groups)]
        st["h2d"] = sum(x.numel() * 2 for x in st["hin"])
        st["d2h"] = sum(x.numel() * 2 for x in st["hout"])
        return st

    E2E_GROUP = 8  # steps per cross-stream synchronisation

    def e2e_run(self, st, stream):
        """All the steps end to end (the caches must hold the fill only: call rewind first)."""
        import torch
        n = self.steps
        groups = [range(g, min(n, g + self.E2E_GROUP)) for g in range(0, n, self.E2E_GROUP)]
        st["copy"].wait_stream(stream)
        with torch.cuda.stream(st["copy"]):
            for gi, grp in enumerate(groups):
                for t in grp:
                    st["din"][t].copy_(st["hin"][t], non_blocking=True)
                st["ev_in"][gi].record(st["copy"])
        for gi, grp in enumerate(groups):
            stream.wait_event(st["ev_in"][gi])
            for t in grp:
                for fn, args in st["calls"][t]:
                    if fn(*args) != 0:
                        raise RuntimeError("vst_dec_step failed")
            st["ev_out"][gi].record(stream)
        with torch.cuda.stream(st["back"]):
            for gi, grp in enumerate(groups):
                st["back"].wait_event(st["ev_out"][gi])
                for t in grp:
                    st["hout"][t].copy_(st["dout"][t], non_blocking=True)
        stream.wait_stream(st["back"])

    def kv_bytes(self, start_positions):
        """Algorithmic bytes of kernel (c) for one run of the steps starting at the given
        positions: K and V of every visible key (min(pos+1, W) keys x Hk x D x 2 B x 2)
        plus the step's q, k, v and out."""
        per_key = DEC_HK * DEC_D * 2 * 2
        io = (DEC_H * DEC_D * 2) * 2 + DEC_HK * DEC_D * 2 * 2
        tot = 0
        for p0 in start_positions:
            for t in range(self.steps):
                tot += min(p0 + t + 1, DEC_W) * per_key + io
        return tot * self.L

    def close(self):
        for row in self.ctxs:
            for c in row:
                c.close()
        self.module.close()


class PrefillWorkload:
    """26 decoder layers of one stream, each prefilling `tokens` prompt tokens on an empty
    cache (vst_dec_prefill per layer). The ring is cleared once before the captured run, and
    a replay redoes the same positions."""

    def __init__(self, spec, dev, rank=0):
        import torch
        from sliding_window_kv_gb300 import synth, vst
        self.vst = vst
        self.L, self.n = spec["layers"], spec["tokens"]
        seed = rank_seed(spec["seed"], rank)
        self.module = vst.Module(vst.DEC)
        self.ctxs = [vst.Ctx(self.module) for _ in range(self.L)]
        self.Q = [synth.frames(synth.tensor_key(seed, 0, l, 0), 0, self.n, DEC_H, DEC_D, dev) for l in range(self.L)]
        self.K = [synth.frames(synth.tensor_key(seed, 0, l, 1), 0, self.n, DEC_HK, DEC_D, dev) for l in range(self.L)]
        self.V = [synth.frames(synth.tensor_key(seed, 0, l, 2), 0, self.n, DEC_HK, DEC_D, dev) for l in range(self.L)]
        self.O = [torch.empty_like(q) for q in self.Q]

    def reset(self, stream):
        for c in self.ctxs:
            self.vst.ctx_reset(c.handle, stream)

    def run(self, stream):
        for l in range(self.L):
            self.vst.dec_prefill(self.ctxs[l].handle, self.Q[l], self.K[l], self.V[l], self.O[l], self.n, stream)

    def kv_bytes(self):
        """Algorithmic bytes of kernel (c) for one run: what n one-token steps read (K and V
        of every visible key, min(p+1, W) keys x Hk x D x 2 B x 2, plus each token's q, k,
        v and out)."""
        per_key = DEC_HK * DEC_D * 2 * 2
        io = (DEC_H * DEC_D * 2) * 2 + DEC_HK * DEC_D * 2 * 2
        return self.L * sum(min(p + 1, DEC_W) * per_key + io for p in range(self.n))

    def close(self):
        for c in self.ctxs:
            c.close()
        self.module.close()


class OfflineWorkload:
    """32 encoder layers over B whole clips of T frames (vst_enc_offline per layer, one plan
    shared by the layers). Inputs of layer l are [B][T][H][D] buffers."""

    def __init__(self, spec, dev, rank=0):
        import torch
        from sliding_window_kv_gb300 import synth, vst
        self.vst = vst
        self.L, self.B, self.T = spec["layers"], spec["clips"], spec["frames"]
        self.left, self.right = spec["left"], spec["right"]
        seed = rank_seed(spec["seed"], rank)
        self.module = vst.Module(vst.ENC)
        self.plan = vst.Offline(self.module, self.B, self.T)
        mk = lambda l, i: torch.stack([synth.frames(synth.tensor_key(seed, b, l, i), 0, self.T, ENC_H, ENC_D, dev)
                                       for b in range(self.B)])
        self.Q = [mk(l, 0) for l in range(self.L)]
        self.K = [mk(l, 1) for l in range(self.L)]
        self.V = [mk(l, 2) for l in range(self.L)]
        self.O = [torch.empty_like(q) for q in self.Q]

    def run(self, stream):
        for l in range(self.L):
            self.plan.run(self.Q[l], self.K[l], self.V[l], self.O[l], self.left, self.right, stream)

    def flops_per_launch(self):
        """4·D FLOP per visible (query, key) pair per head, for one layer of all clips."""
        T, L, R = self.T, self.left, max(self.right - 1, 0)
        pairs = sum(min(i, L - 1) + 1 + min(R, T - 1 - i) for i in range(T))
        return 4.0 * ENC_D * pairs * ENC_H * self.B

    def close(self):
        self.plan.close()
        self.module.close()


# ---------------------------------------------------------------- timing helpers

def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        fn(torch.cuda.current_stream())
    return g


def time_graph(g, stream, n, dist=None):
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(n):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return a.elapsed_time(b)


def profiled_kernels(step_fn, stream):
    """Capture one step with per-kernel events on, replay it twice, return the second
    replay's {kernel: (launches, total_ms)}."""
    import torch
    from sliding_window_kv_gb300 import vst
    vst.prof_read()
    vst.prof_enable(True)
    try:
        g = capture(step_fn, stream)
    finally:
        vst.prof_enable(False)
    g.replay()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    return vst.prof_read()


def region_launch_us(prof, kernel, region_ms):
    """Average duration of one launch of `kernel` inside the timed region: the region's time
    (CUDA events around the replayed step) split between kernels in proportion to their
    per-launch event totals from the profiled replay, divided by the kernel's launches.
    Kernels of a step overlap their neighbours (programmatic dependent launch) in the timed
    region; the profiled replay brackets each launch with events and so loses that overlap."""
    nl, kms = prof[kernel]
    total = sum(v[1] for v in prof.values() if v[0])
    return 1e3 * region_ms * (kms / total) / nl


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


TIMING_NOTE = ("avg_launch_us: timed region / launches, split between kernels by their profiled event "
               "shares; isolated_launch_us: events around each launch (no overlap with neighbours)")

# sources of each profiled kernel id (the encoder attention id covers all its launch shapes)
_COMMON_SOURCES = ("ptx.cuh", "common.cuh", "vst_internal.h")
KERNEL_SOURCES = {"enc_attn_kernel": ("enc_attn.cu", "enc_attn_split.cu", "enc_common.cuh") + _COMMON_SOURCES,
                  "dec_step_kernel": ("dec_step.cu",) + _COMMON_SOURCES, "compact_kernel": ("compact.cu",) + _COMMON_SOURCES}


def kernel_source_sha(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "sliding_window_kv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str, units_per_launch: float, workload: str = "", fallback: bool = True):
    """DRAM bytes (read + write) per launch from the committed ncu capture, scaled from the
    captured case to this launch by the work units it processes; None when there is no
    capture or the kernel's source changed since it was taken. A capture of the workload's
    own launch shape ("kernel@workload") is preferred to the kernel's default one, which is
    used only when `fallback` (the same launch shape)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        t = json.load(open(p))
        d = t.get("%s@%s" % (kernel, workload)) or (t.get(kernel) if fallback else None)
        if not d or d.get("source_sha") != kernel_source_sha(kernel):
            return None
        return d["dram_bytes_per_unit"] * units_per_launch
    except Exception:
        return None


# ---------------------------------------------------------------- CPU baseline (oracle)

def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline_enc(spec, layers_sample: int, threads: int):
    """Time the fp64 oracle on `layers_sample` layers of stream 0 of the workload (whole
    clip per layer) and scale to encoder frames/s of the full workload."""
    import oracle
    from sliding_window_kv_gb300 import synth
    n = spec["frames"]
    seed = spec["seed"]
    ins = []
    for l in range(layers_sample):
        ins.append([synth.bits(synth.frames(synth.tensor_key(seed, 0, l, i), 0, n, ENC_H, ENC_D)) for i in range(3)])
    t0 = time.perf_counter()
    for q, k, v in ins:
        oracle.attention(q, k, v, ENC_W, threads=threads)
    dt = time.perf_counter() - t0
    per_layer = dt / layers_sample
    fps = n / (per_layer * spec["layers"])
    return fps, dt, "oracle on %d of %d layers, whole %d-frame clip of stream 0, %d threads" % (
        layers_sample, spec["layers"], n, threads)


def cpu_baseline_dec(spec, steps_sample: int, threads: int):
    """Time the oracle for `steps_sample` decoder steps of one layer at a full 8192 window
    and scale to decoder steps/s of the 26-layer step."""
    import numpy as np

    import oracle
    from sliding_window_kv_gb300 import synth
    seed = spec["seed"]
    fill = DEC_W
    n = fill + steps_sample
    q = synth.bits(synth.frames(synth.tensor_key(seed, 0, 0, 0), 0, n, DEC_H, DEC_D))
    k = synth.bits(synth.frames(synth.tensor_key(seed, 0, 0, 1), 0, n, DEC_HK, DEC_D))
    v = synth.bits(synth.frames(synth.tensor_key(seed, 0, 0, 2), 0, n, DEC_HK, DEC_D))
    t0 = time.perf_counter()
    qr = np.zeros((n, DEC_H, DEC_D))
    qr[fill:] = oracle.rope_rows(q[fill:], fill)
    kr = oracle.rope_rows(k, 0)
    vv = oracle.bf16_to_double(v)
    oracle.attend(qr, kr, vv, DEC_W, rows=(fill, n), threads=threads)
    dt = time.perf_counter() - t0
    sps = steps_sample / (dt * spec["layers"])
    return sps, dt, "oracle on 1 of %d layers, %d steps at window 8192 (incl. RoPE of the window), %d threads" % (
        spec["layers"], steps_sample, threads)


# ---------------------------------------------------------------- arms

def run_reference(args, dist):
    """The oracle as it stands, on this host's cores, over a bounded sample per step."""
    if dist.rank != 0:
        return
    spec = WORKLOADS[args.workload]
    threads = cpu_threads()
    vals = []
    for i in range(args.warmup + args.steps):
        if spec["kind"] == "enc":
            v, dt, sample = cpu_baseline_enc(spec, 1, threads)
        else:
            v, dt, sample = cpu_baseline_dec(spec, 8, threads)
        if i >= args.warmup:
            vals.append((v, dt))
    total = sum(dt for _, dt in vals)
    value = statistics.mean(v for v, _ in vals)
    unit = "enc frames/s" if spec["kind"] == "enc" else "dec steps/s"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / max(1, len(vals)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args.workload, spec),
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def workload_config(name, spec):
    if spec["kind"] == "enc":
        return {"workload": "enc_%dL_%dx%d_W%d_ring1536_%dstream_%dframes_chunk%d%s" % (
            spec["layers"], ENC_H, ENC_D, ENC_W, spec["streams"], spec["frames"], spec["feed"],
            "_stagger%d" % spec["stagger"] if spec["stagger"] else ""),
            "layers": spec["layers"], "streams": spec["streams"], "frames_per_stream": spec["frames"],
            "chunk": spec["feed"], "seed": spec["seed"],
            "l2": "inputs larger than L2 (no flush)"}
    return {"workload": "dec_%dL_gqa%d-%dx%d_W%d_%dstreams_fill_%s_steps%d" % (
        spec["layers"], DEC_H, DEC_HK, DEC_D, DEC_W, spec["streams"], spec["fill"], spec["steps"]),
        "layers": spec["layers"], "streams": spec["streams"], "steps": spec["steps"], "seed": spec["seed"],
        "l2": "KV cache read per step larger than L2 (no flush)"}


def bench_dec(spec, dev, stream, dist, n_steps, warmup, peaks, want_cpu, e2e=False, workload="dec_b1"):
    import torch
    from sliding_window_kv_gb300 import vst
    w = DecWorkload(spec, dev, n_steps, dist.rank)
    w.run_steps(stream)  # eager warm-up (also configures kernels)
    torch.cuda.synchronize()
    n0 = vst.launch_count()
    g = capture(w.run_steps, stream)
    launches = vst.launch_count() - n0
    for _ in range(max(1, warmup)):
        g.replay()
    steps_per_s, ms = dist.job_rate(w.steps, time_graph(g, stream, 1, dist))
    start_pos = w.positions()
    prof = profiled_kernels(w.run_steps, stream)
    nl, kms = prof["dec_step_kernel"]
    bytes_per_launch = w.kv_bytes(start_pos) / max(1, nl)
    launch_us = region_launch_us(prof, "dec_step_kernel", ms)
    achieved = bytes_per_launch / (launch_us / 1e6) / 1e9
    hbm, _, _, src = peaks
    out = {"value": steps_per_s, "unit": "dec steps/s", "config": workload_config("", spec),
           "ms_per_step": ms / w.steps, "gpu_launches": launches,
           "roofline": {"kernel": "dec_step_kernel", "bound": "hbm", "achieved": achieved, "peak": hbm,
                        "unit": "GB/s", "frac": achieved / hbm,
                        "traffic": dram_traffic("dec_step_kernel", bytes_per_launch, workload,
                                                fallback=workload == "dec_b1"),
                        "peak_source": src, "launches": nl, "avg_launch_us": launch_us,
                        "isolated_launch_us": 1e3 * kms / nl, "timing": TIMING_NOTE,
                        "algorithmic_bytes_per_launch": bytes_per_launch}}
    if e2e:
        # the same steps through the C ABI with host copies: the eager, captured and profiled
        # runs above advanced each context's position on the host, and the e2e run steps on
        # from there (at a full window every step reads the same number of keys)
        est = w.e2e_setup(stream)
        w.e2e_run(est, stream)  # warm-up
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        a.record(stream)
        w.e2e_run(est, stream)
        b.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        dist.barrier()
        e2e_value, _ = dist.job_rate(w.steps, a.elapsed_time(b))
        calls = [c for t in est["calls"] for c in t]  # the steps once more, timed on the host alone
        host_ms, host_us = host_enqueue_cost(calls)
        out["e2e"] = {"value": e2e_value, "unit": "dec steps/s",
                      "h2d_bytes_per_step": est["h2d"] / w.steps, "d2h_bytes_per_step": est["d2h"] / w.steps,
                      "steps": w.steps, "host_wall_s": wall,
                      "host_enqueue_ms_per_step": host_ms / w.steps, "host_us_per_call": host_us,
                      "calls_per_step": len(calls) / w.steps,
                      "path": "vst_dec_step per layer and step through the C ABI (no graph); each step's inputs "
                              "(all layers) copied host to device in one copy on a copy stream, its outputs back "
                              "on a third stream, one cross-stream wait per 8 steps, pinned memory, all inside "
                              "the region"}
        del est
    if want_cpu:
        # the oracle on one stream at a full window, scaled to the workload's streams and
        # their mean visible keys per step (its time per step is linear in the keys)
        v, dt, sample = cpu_baseline_dec(spec, 16, cpu_threads())
        v1, dt1, sample1 = cpu_baseline_dec(spec, 4, 1)
        keys = statistics.mean(min(p + t + 1, DEC_W) for p in start_pos for t in range(w.steps)) * len(start_pos)
        scale = DEC_W / keys
        out["cpu_baseline"] = {"value": v * scale, "unit": "dec steps/s", "cores": cpu_threads(), "kind": "oracle",
                               "sample": sample + ("; scaled to %d streams of %.0f visible keys on average"
                                                   % (len(start_pos), keys / len(start_pos)) if scale != 1 else ""),
                               "seconds": dt,
                               "single_thread": {"value": v1 * scale, "sample": sample1, "seconds": dt1}}
    w.close()
    return out


def bench_offline(spec, dev, stream, dist, steps, warmup, peaks):
    import torch
    from sliding_window_kv_gb300 import vst
    w = OfflineWorkload(spec, dev, dist.rank)
    w.run(stream)  # eager warm-up (configures the kernels)
    torch.cuda.synchronize()
    n0 = vst.launch_count()
    g = capture(w.run, stream)
    launches = vst.launch_count() - n0
    for _ in range(max(1, warmup)):
        g.replay()
    frames_per_s, ms = dist.job_rate(w.B * w.T * steps, time_graph(g, stream, steps, dist))
    ms /= steps  # per pass of all layers
    prof = profiled_kernels(w.run, stream)
    nl, kms = prof["enc_attn_kernel"]
    flops = w.flops_per_launch()
    launch_us = region_launch_us(prof, "enc_attn_kernel", ms)
    achieved = flops / (launch_us / 1e6) / 1e12
    _, tflops, _, src = peaks
    out = {"value": frames_per_s, "unit": "enc frames/s",
           "config": {"workload": "enc_offline_%dL_20x64_%dclips_%dframes_left%d_right%d" % (w.L, w.B, w.T, w.left, w.right),
                      "layers": w.L, "clips": w.B, "frames_per_clip": w.T, "left": w.left, "right": w.right,
                      "seed": spec["seed"], "l2": "inputs larger than L2 (no flush)"},
           "ms_per_step": ms, "gpu_launches": launches,
           "roofline": {"kernel": "enc_attn_kernel", "bound": "tensor", "achieved": achieved, "peak": tflops,
                        "unit": "TFLOP/s", "frac": achieved / tflops,
                        "traffic": dram_traffic("enc_attn_kernel", flops, "enc_offline%d" % w.B + ("_la" if w.right else ""),
                                                fallback=False),
                        "peak_source": src, "launches": nl, "avg_launch_us": launch_us,
                        "isolated_launch_us": 1e3 * kms / nl, "timing": TIMING_NOTE,
                        "algorithmic_flops_per_launch": flops},
           "kernels": {k: {"launches": v[0], "total_ms": v[1]} for k, v in prof.items()}}
    w.close()
    return out


def bench_prefill(spec, dev, stream, dist, steps, warmup, peaks):
    import torch
    from sliding_window_kv_gb300 import vst
    w = PrefillWorkload(spec, dev, dist.rank)
    w.run(stream)  # eager: allocates each ctx's prefill scratch, configures the kernels
    w.reset(stream)
    torch.cuda.synchronize()
    n0 = vst.launch_count()
    g = capture(w.run, stream)
    launches = vst.launch_count() - n0
    for _ in range(max(1, warmup)):
        g.replay()
    tok_per_s, ms = dist.job_rate(w.n * steps, time_graph(g, stream, steps, dist))
    ms /= steps  # per run of the 26 layers
    w.reset(stream)
    prof = profiled_kernels(w.run, stream)
    nl, kms = prof["dec_step_kernel"]
    bytes_per_launch = w.kv_bytes() / max(1, nl)
    launch_us = region_launch_us(prof, "dec_step_kernel", ms)
    achieved = bytes_per_launch / (launch_us / 1e6) / 1e9
    hbm, _, _, src = peaks
    out = {"value": tok_per_s, "unit": "prompt tokens/s",
           "config": {"workload": "dec_prefill_%dL_gqa32-8x128_W8192_1stream_%dtok" % (w.L, w.n), "layers": w.L,
                      "tokens": w.n, "seed": spec["seed"], "l2": "prompt K/V fit in L2 (no flush between replays)"},
           "ms_per_step": ms, "gpu_launches": launches,
           "roofline": {"kernel": "dec_step_kernel", "bound": "hbm", "achieved": achieved, "peak": hbm,
                        "unit": "GB/s", "frac": achieved / hbm,
                        "traffic": dram_traffic("dec_step_kernel", bytes_per_launch, "dec_prefill%d" % w.n, fallback=False),
                        "peak_source": src, "launches": nl, "avg_launch_us": launch_us,
                        "isolated_launch_us": 1e3 * kms / nl, "timing": TIMING_NOTE,
                        "algorithmic_bytes_per_launch": bytes_per_launch}}
    w.close()
    return out


def bench_enc(spec, dev, stream, dist, steps, warmup, peaks, workload, e2e=True, want_cpu=False):
    """One encoder streaming workload: `value` from CUDA-graph replays of the step, the
    attention's roofline, the compaction's HBM fraction and (e2e) the same step through the
    C ABI with host copies inside the region."""
    import torch
    from sliding_window_kv_gb300 import vst
    w = EncWorkload(spec, dev, dist.rank)
    w.run_step(stream)  # eager warm-up
    torch.cuda.synchronize()
    n0 = vst.launch_count()
    g = capture(w.run_step, stream)
    launches_per_step = vst.launch_count() - n0
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    value, ms = dist.job_rate(w.frames_per_step * steps, time_graph(g, stream, steps, dist))
    prof = profiled_kernels(w.run_step, stream)
    del g

    # dominant kernel: chunk attention (kernel b), tensor-bound
    nl, kms = prof["enc_attn_kernel"]
    flops_per_launch = w.attn_flops() / max(1, nl)
    launch_us = region_launch_us(prof, "enc_attn_kernel", ms / steps)
    achieved = flops_per_launch / (launch_us / 1e6) / 1e12
    hbm, tf, tfs, src = peaks
    out = {"value": value, "unit": "enc frames/s", "ms_per_step": ms / steps,
           "config": workload_config(workload, spec),
           "roofline": {"kernel": "enc_attn_kernel", "bound": "tensor", "achieved": achieved, "peak": tf,
                        "unit": "TFLOP/s", "frac": achieved / tf,
                        "traffic": dram_traffic("enc_attn_kernel", flops_per_launch, workload),
                        "peak_source": src + " bf16 burst", "launches": nl,
                        "avg_launch_us": launch_us, "isolated_launch_us": 1e3 * kms / nl,
                        "timing": TIMING_NOTE, "algorithmic_flops_per_launch": flops_per_launch},
           "kernels": {k: {"launches": v[0], "total_ms": v[1]} for k, v in prof.items() if v[0]},
           "gpu_launches": launches_per_step * steps}
    ncmp, cms = prof["compact_kernel"]
    if ncmp:
        cb = w.compact_bytes() / ncmp
        cus = region_launch_us(prof, "compact_kernel", ms / steps)
        out["compaction"] = {"kernel": "compact_kernel", "bound": "hbm", "launches": ncmp,
                             "avg_launch_us": cus, "isolated_launch_us": 1e3 * cms / ncmp,
                             "timing": TIMING_NOTE, "algorithmic_bytes_per_launch": cb,
                             "achieved_gbs": cb / (cus / 1e6) / 1e9, "frac": cb / (cus / 1e6) / 1e9 / hbm,
                             "traffic": dram_traffic("compact_kernel", cb, workload, fallback=workload == "enc_stream")}

    if e2e:
        est = w.e2e_setup(stream)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        w.e2e_run(est, stream)  # warm-up
        torch.cuda.synchronize()
        e2e_steps = max(1, min(steps, 5))
        dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        a.record(stream)
        for _ in range(e2e_steps):
            w.e2e_run(est, stream)
        b.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        dist.barrier()
        e2e_value, _ = dist.job_rate(w.frames_per_step * e2e_steps, a.elapsed_time(b))
        # one more step's calls (context resets first), timed on the host alone
        calls = list(est["resets"]) + [c for f in est["calls"] for c in f]
        host_ms, host_us = host_enqueue_cost(calls)
        n_calls = len(calls)
        out["e2e"] = {"value": e2e_value, "unit": "enc frames/s",
                      "h2d_bytes_per_step": est["h2d"], "d2h_bytes_per_step": est["d2h"],
                      "steps": e2e_steps, "host_wall_s": wall,
                      "host_enqueue_ms_per_step": host_ms, "host_us_per_call": host_us, "calls_per_step": n_calls,
                      "path": "vst_enc_feed per layer and feed through the C ABI (no graph); each feed's "
                              "inputs copied host to device in one copy on a copy stream, its outputs back "
                              "on a third stream, one cross-stream wait per 8 feeds, pinned memory, all "
                              "inside the region"}
        del est
    w.close()
    if want_cpu:
        v, dt, sample = cpu_baseline_enc(spec, 1, cpu_threads())
        out["cpu_baseline"] = {"value": v, "unit": "enc frames/s", "cores": cpu_threads(), "kind": "oracle",
                               "sample": sample, "seconds": dt}
    return out


def run_vst(args, dist):
    import torch
    from sliding_window_kv_gb300 import vst
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the benchmark needs the GPU (there is no CPU path)")
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    vst.lib()
    stream = torch.cuda.Stream(dev)
    peaks = load_peaks()
    spec = dict(WORKLOADS[args.workload])
    if args.layers:
        spec["layers"] = args.layers
    if spec["kind"] == "dec":
        spec["steps"] = args.dec_steps
    sampler = ClockSampler(dist.local_rank)
    line = {"metric": METRIC, "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded counter-hash bf16 ~N(0,1))", "impl": "vst"}

    if spec["kind"] == "offline":
        with torch.cuda.stream(stream):
            sampler.start()
            d = bench_offline(spec, dev, stream, dist, args.steps, args.warmup, peaks)
            clocks = sampler.stop()
        line.update({"value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"], "config": d["config"],
                     "roofline": d["roofline"], "gpu_launches": d["gpu_launches"], "kernels": d["kernels"],
                     "clocks": clocks})
        if dist.rank == 0:
            print(json.dumps(line))
        return

    if spec["kind"] == "prefill":
        with torch.cuda.stream(stream):
            sampler.start()
            d = bench_prefill(spec, dev, stream, dist, args.steps, args.warmup, peaks)
            clocks = sampler.stop()
        line.update({"value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"], "config": d["config"],
                     "roofline": d["roofline"], "gpu_launches": d["gpu_launches"], "clocks": clocks})
        if dist.rank == 0:
            print(json.dumps(line))
        return

    if spec["kind"] == "dec":
        with torch.cuda.stream(stream):
            sampler.start()
            d = bench_dec(spec, dev, stream, dist, spec["steps"], args.warmup, peaks, want_cpu_baseline(args, dist),
                          e2e=not args.no_e2e, workload=args.workload)
            clocks = sampler.stop()
        line.update({"value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"], "config": d["config"],
                     "roofline": d["roofline"], "gpu_launches": d["gpu_launches"], "clocks": clocks})
        for k in ("cpu_baseline", "e2e"):
            if k in d:
                line[k] = d[k]
        if dist.rank == 0:
            print(json.dumps(line))
        return

    with torch.cuda.stream(stream):
        sampler.start()
        d = bench_enc(spec, dev, stream, dist, args.steps, args.warmup, peaks, args.workload, e2e=not args.no_e2e)
        clocks = sampler.stop()
        line.update({k: v for k, v in d.items() if k != "clocks"})
        line["clocks"] = clocks

        if not args.no_dec and args.workload == "enc_stream":
            # the other configurations of the metric, each an object of the line: the decoder
            # at batch 1 (with its end-to-end figure), 64 decoder streams, 16 encoder streams
            # in 512-frame batches, and the next rows (prefill, offline encoder)
            def timed(fn):
                smp = ClockSampler(dist.local_rank)
                smp.start()
                out = fn()
                out["clocks"] = smp.stop()
                torch.cuda.empty_cache()
                return out

            dspec = dict(WORKLOADS["dec_b1"])
            dspec["steps"] = args.dec_steps
            line["dec"] = timed(lambda: bench_dec(dspec, dev, stream, dist, args.dec_steps, args.warmup, peaks,
                                                  want_cpu_baseline(args, dist), e2e=not args.no_e2e))
            dspec64 = dict(WORKLOADS["dec_b64"])
            dspec64["steps"] = args.dec_steps
            line["dec_b64"] = timed(lambda: bench_dec(dspec64, dev, stream, dist, args.dec_steps, args.warmup, peaks,
                                                      want_cpu_baseline(args, dist), workload="dec_b64"))
            line["enc_long16"] = timed(lambda: bench_enc(dict(WORKLOADS["enc_long16"]), dev, stream, dist,
                                                         args.steps, args.warmup, peaks, "enc_long16", e2e=False,
                                                         want_cpu=want_cpu_baseline(args, dist)))
            line["prefill"] = timed(lambda: bench_prefill(dict(WORKLOADS["dec_prefill39"]), dev, stream, dist,
                                                          args.steps, args.warmup, peaks))
            line["offline"] = timed(lambda: bench_offline(dict(WORKLOADS["enc_offline4"]), dev, stream, dist,
                                                          args.steps, args.warmup, peaks))

    if want_cpu_baseline(args, dist):
        v, dt, sample = cpu_baseline_enc(spec, 4 if spec["layers"] >= 4 else spec["layers"], cpu_threads())
        v1, dt1, sample1 = cpu_baseline_enc(spec, 1, 1)
        line["cpu_baseline"] = {"value": v, "unit": "enc frames/s", "cores": cpu_threads(), "kind": "oracle",
                                "sample": sample, "seconds": dt,
                                "single_thread": {"value": v1, "sample": sample1, "seconds": dt1}}
    if dist.rank == 0:
        print(json.dumps(line))


def main():
    args = parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if world > 1 and rank != 0:
            return
        class _D:
            rank = 0
        run_reference(args, _D())
        return
    dist = Dist(args.gpus)
    try:
        run_vst(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
