"""Host-side logic of bench.py on the CPU: the multi-rank reduction over two gloo ranks, and the
reference arm (the CPU oracle) printing its one JSON line."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, lr, w = bench.dist_env()
    assert (r, lr, w) == (rank, rank, world)
    bench.init_dist(w, "gloo")
    # rank r took (r + 1) seconds for 10 units: the job is 20 units over the slowest 2 s
    value, tmax = bench.aggregate(10.0, float(r + 1), w)
    m = bench.reduce_max(3.0 * r, w)
    bench.barrier(w)
    q.put((rank, value, tmax, m))
    dist.destroy_process_group()


def test_two_rank_aggregate():
    import socket
    import torch.multiprocessing as mp
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, tmax, m in got:
        assert tmax == 2.0 and value == 10.0 and m == 3.0


def test_single_rank_defaults():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.5, 1) == 1.5
    assert bench.aggregate(8.0, 2.0, 1) == (4.0, 2.0)


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_baseline_reports_threads_and_one_core():
    """The bench line's CPU baseline: the oracle on every host core and on one, with the CPU named."""
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    d = bench.cpu_baseline(argparse.Namespace(cpu_seconds=0.3))
    assert d["kind"] == "oracle" and d["unit"] == "GB/s" and d["cores"] >= 1 and d["value"] > 0
    assert d["one_thread"]["value"] > 0 and d["one_thread"]["unit"] == "GB/s"
    assert isinstance(d["cpu"], str) and d["cpu"]
