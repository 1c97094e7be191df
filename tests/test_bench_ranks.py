"""The multi-rank host logic of bench.py on the CPU (gloo, world size 2).

The layer shards as independent replicas, so the only cross-rank steps are
the barriers around the timed region, the max over ranks of the step time,
and the whole-job value; the reference arm runs on rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        barrier, max_over_ranks = bench.rank_ops(dist, world, "cpu")
        barrier()
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
        ms = max_over_ranks(local_ms)
        out.put((rank, ms, bench.decode_value(ms, 16, world)))
        barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; the value divides it by the
    # tokens of both ranks: 15 ms / (16 layers x 2 ranks) = 468.75 µs
    assert [r[1] for r in res] == [15.0, 15.0]
    assert [r[2] for r in res] == [468.75, 468.75]


def test_single_process_ops_are_plain():
    barrier, max_over_ranks = bench.rank_ops(None, 1, "cpu")
    barrier()
    assert max_over_ranks(3.5) == 3.5
    assert bench.decode_value(2.0, 16, 1) == 125.0


def test_reference_arm_under_torchrun_prints_on_rank_0_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
