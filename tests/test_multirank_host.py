"""Host logic of bench.py's N > 1 path on CPU with two gloo ranks.

Under torchrun every rank runs its own seeded problem (weak scaling) and
rank 0 reports the maximum time over ranks.  This checks the max reduction,
the barrier and the per-rank input seeding without a GPU.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    from newton_schulz_nesterov_gb300 import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        w = bench.rank_workload("tinymlp_d128", rank)
        g = workloads.grad(w, 0, 0)
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, torch.tensor([float(g.double().sum())], dtype=torch.float64))
        out[rank] = (got, [float(x) for x in sums], w.shapes == workloads.get("tinymlp_d128").shapes)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_seeding():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        got, sums, same_shapes = out[r]
        assert got == 15.0              # max over ranks of 10 + 5*rank
        assert same_shapes              # same problem shapes on every rank
        assert sums[0] != sums[1]       # but independent seeded inputs


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.rank_workload("tinymlp_d128", 0).seed == 1235
