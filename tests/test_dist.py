"""The multi-GPU path of bench.py at world size 2, on CPU with the gloo backend.

The path shards by streams with no exchange step: under torchrun every rank runs an
independent replica on its own seeded inputs (weak scaling), the timed region is bracketed
by barriers, and the whole-job value is all ranks' units over the slowest rank's time. The
reference arm (the oracle) runs on rank 0 alone; the other ranks exit 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, port, ms_local, out):
    os.environ.update(WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    from sliding_window_kv_gb300 import synth
    d = bench.Dist(2)
    try:
        d.barrier()
        value, ms = d.job_rate(1000 * 4, ms_local[rank])
        d.barrier()
        seed = bench.rank_seed(2, rank)
        first = synth.frames(synth.tensor_key(seed, 0, 0, 0), 0, 2, 20, 64, "cpu")
        out.put((rank, d.world, value, ms, seed, first.view(-1)[:8].tolist()))
    finally:
        d.close()


def test_replicas_report_all_units_over_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    ms_local = [10.0, 25.0]
    procs = [ctx.Process(target=_replica, args=(r, port, ms_local, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, world, value, ms, _, _ in res:
        assert world == 2
        assert ms == 25.0                          # the slowest rank's time, on every rank
        assert value == 2 * 1000 * 4 / 0.025       # both ranks' units over that time
    # each replica streams its own inputs
    assert res[0][4] != res[1][4]
    assert res[0][5] != res[1][5]


def test_reference_arm_prints_once_under_torchrun():
    """bench.py --impl reference on two ranks: one JSON line, from rank 0; both exit 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "enc_small", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
