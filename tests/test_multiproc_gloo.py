"""The benchmark's multi-process logic on CPU with the gloo backend, world size
2: every rank runs its own replica (no collective on the data path); the step
time is the maximum over ranks and the job value counts the work of every rank.
The reference arm prints from rank 0 only."""
import os
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    local_ms = [3.0, 5.5][rank]
    m = bench.max_over_ranks(local_ms, world, "cpu")
    v = bench.job_throughput(1e12, m, world)
    dist.barrier()
    out[rank] = (m, v)
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world = 2
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        m, v = res[rank]
        assert m == 5.5                               # the slowest replica
        assert abs(v - 2 * 1e12 / 5.5e-3 / 1e12) < 1e-9  # both replicas' work


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
