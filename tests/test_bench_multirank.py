"""The bench's multi-process path on CPU: two gloo ranks agree on the slowest
rank's time and on the whole-job throughput (weak scaling: every rank moves
its own bytes); the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (world, rank, rank)
    ms, gbs = bench.aggregate(10.0 * (rank + 1), 1e9, world)
    bench.barrier()
    out[rank] = (ms, gbs)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_bytes():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, gbs = res[rank]
        assert ms == pytest.approx(20.0)                      # the slowest rank
        assert gbs == pytest.approx(world * 1e9 / 0.020 / 1e9)  # bytes of both ranks


def test_reference_arm_only_on_rank_zero():
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=3)
    assert bench.run_reference(args, world=2, rank=1) is None


def test_single_process_aggregate_is_identity():
    import bench
    ms, gbs = bench.aggregate(4.0, 8e9, 1)
    assert ms == 4.0 and gbs == pytest.approx(2000.0)
