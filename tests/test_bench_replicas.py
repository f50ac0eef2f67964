"""The benchmark's multi-GPU mode runs independent replicas (the output
tiles shard without any exchange, and every box here has one GPU).  Its
host-side combination -- barrier, max of the per-rank times, whole-job
throughput -- is checked with two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench  # noqa: PLC0415
    dist.barrier()
    mine = 100.0 + 25.0 * rank            # rank 1 is the slow one
    slowest = bench.max_over_ranks(mine)
    value = bench.job_value(1e12, 4, world, slowest)
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_two_replicas_combine_to_the_slowest_rank():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, value = res[0]
    assert slowest == 125.0
    # 2 replicas x 4 steps x 1e12 ops in 0.125 s = 64 TOPS
    assert value == pytest.approx(64.0)


def test_single_process_is_identity():
    import bench  # noqa: PLC0415
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(2e12, 5, 1, 1000.0) == pytest.approx(10.0)
