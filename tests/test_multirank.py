"""Multi-process host logic of bench.py on the CPU (gloo, world size 2): the
whole-job value is every rank's work over the slowest rank's time, and the
reference arm runs on rank 0 only."""
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    m = bench.reduce_max_ms(ms, dist, "cpu")
    out[rank] = (m, bench.whole_job_gbs(1_000_000_000, world, m))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, 29531, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        m, v = res[rank]
        assert m == 5.0                       # the slowest rank's time
        assert v == pytest.approx(2 * 1e9 / 5e-3 / 1e9)  # both ranks' bytes over it


def test_single_process_aggregation():
    assert bench.reduce_max_ms(2.5) == 2.5
    assert bench.whole_job_gbs(6_553_600, 1, 1e-3) == pytest.approx(6553.6)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
