"""Host logic of bench.py that needs no GPU: whole-job aggregation over ranks
(gloo, world size 2, on CPU) and the reference arm's non-zero ranks."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_setup()
    ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms, ws)
    bench.barrier(ws)
    value = bench.aggregate(100.0, ms_max, ws)
    q.put((r, ws, ms_max, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29611
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, ws, ms_max, value in res:
        assert ws == 2
        assert ms_max == 15.0                   # max over ranks
        assert value == pytest.approx(100.0 * 2 / 15e-3)   # units of all ranks / max time


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, env=env,
                         timeout=120)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_oracle_child_reports_flops():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--_oracle-child", "16", "1"],
                         capture_output=True, text=True, timeout=300,
                         env=dict(os.environ, OPENBLAS_NUM_THREADS="2"))
    assert res.returncode == 0, res.stderr
    d = json.loads(res.stdout.strip().splitlines()[-1])
    assert d["tokens"] == 16 and d["flops"] == 6.0 * 16 * 2 * 2048 * 2048
    assert len(d["times"]) == 1 and d["times"][0] > 0
