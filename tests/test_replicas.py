"""The bench on several GPUs: independent replicas.

Sequences share nothing, so each rank runs the whole verify path alone and the
ranks meet only to time it: every rank reports the slowest rank's time, and
the job's rate counts every rank's calls over that time.  Tested here with
two gloo ranks on the CPU (the GPU runs use NCCL for the same one
all-reduce), and the reference arm under torchrun: rank 0 alone runs the
oracle and prints the one line, the other rank leaves at once."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], dist, "cpu")
        q.put((rank, ms, bench.job_rate(40, world, ms / 1e3)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_every_rank_reports_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local_ms = [12.5, 30.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert [g[1] for g in got] == [30.0, 30.0]
    # 40 calls on each of two ranks over the slower rank's 30 ms
    assert all(g[2] == pytest.approx(80 / 0.030) for g in got)


def test_one_rank_needs_no_group():
    assert bench.max_over_ranks(7.0) == 7.0
    assert bench.job_rate(10, 1, 0.5) == 20.0


def test_reference_arm_prints_one_line_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup",
           "0", "--widths", "1"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
