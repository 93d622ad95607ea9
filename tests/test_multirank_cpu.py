"""The multi-GPU path of bench.py on CPU: world_size-2 gloo ranks.

The projection shards only as independent replicas (each GPU runs the whole
load; there is no collective in the data path).  What bench.py does across
ranks is host logic: a barrier around the timed region, the max over ranks
of the per-load time, and rank 0 alone printing the JSON line.  These tests
run that logic on two gloo ranks on the CPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, values, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        mx = bench.max_over_ranks(torch, values[rank], "cpu")
        q.put((rank, mx, bench.whole_job_us_per_load(mx, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_on_two_gloo_ranks():
    world, port = 2, _free_port()
    values = [41.5, 43.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, values, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, mx, job in got:
        assert mx == max(values)  # every rank sees the slowest replica
        assert job == pytest.approx(max(values) / world)


def test_reference_arm_under_torchrun_prints_once(tmp_path):
    """`bench.py --impl reference` launched as two ranks: rank 0 prints one
    JSON line with impl=reference; rank 1 exits 0 without work."""
    pytest.importorskip("numpy")
    from oracle import oracle
    oracle._load()  # the C oracle must be built (build() does it)
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
