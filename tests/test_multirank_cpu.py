"""The multi-rank path of bench.py on CPU: two gloo ranks (world size 2) agree on the slowest
rank's time, the whole-job rate counts every rank's work over that time, and under a torchrun
environment only rank 0 of the reference arm prints its line."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = 10.0 + 5.0 * rank                       # rank 1 is the slowest
    got = bench.max_over_ranks(torch, world, mine, torch.device("cpu"))
    bench.barrier(world)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_whole_job_rate_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1.288e11, 100, 1, 13.0)
    two = bench.whole_job_tflops(1.288e11, 100, 2, 13.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(1.288e11 * 100 / 0.013 / 1e12)


@pytest.mark.parametrize("rank,expect_line", [(0, True), (1, False)])
def test_reference_arm_prints_on_rank0_only(rank, expect_line):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--reference-rows", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if expect_line:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
        assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []
