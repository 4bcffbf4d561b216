"""The multi-process side of bench.py on the host: world size 2 over gloo
(CPU), the same calls the GPU job makes over NCCL.  Each rank runs N
independent replicas' worth of work ("replicas only": the rows of W are
independent, nothing is exchanged on the data path), so the only
collective is the timing reduction."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, dist, "cpu")
    value = bench.job_throughput(1000.0, slowest, world)
    dist.barrier()
    dist.destroy_process_group()
    with open(out, "w") as f:
        json.dump({"rank": rank, "slowest": slowest, "value": value}, f)


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    outs = [str(tmp_path / f"r{r}.json") for r in range(2)]
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, 2, port, outs[r])) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = [json.load(open(o)) for o in outs]
    assert [r["slowest"] for r in res] == [15.0, 15.0]
    # 1000 units per rank per step, two ranks, 15 ms per step -> 133333.3 units/s
    assert all(abs(r["value"] - 2000.0 / 0.015) < 1e-6 for r in res)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.job_throughput(1e9, 1.0, 1) == pytest.approx(1e12)


def test_reference_arm_prints_only_on_rank_0():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
