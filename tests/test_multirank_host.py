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


def test_gpus_flag_starts_ranks_through_torchrun():
    """`bench.py --gpus N` without a launcher reruns itself under torchrun
    with N ranks on 127.0.0.1 and the same arguments; under a launcher the
    world size must match --gpus."""
    import bench
    cmd = bench.spawn_command(4, ["--gpus", "4", "--steps", "2"], 29555)
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=4" in cmd and cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index("--master-port") + 1] == "29555"
    assert cmd[-5].endswith("bench.py") and cmd[-4:] == ["--gpus", "4", "--steps", "2"]


def test_gpus_flag_and_world_size_must_agree(monkeypatch):
    import sys
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4"])
    with pytest.raises(SystemExit):
        bench.main()


def test_cpu_baseline_sample_covers_every_shape():
    """The CPU baseline times one matrix per distinct shape of the workload
    and scales each by its count: for the Llama-3-8B set q, k (= v),
    gate (= up) and down, 32 of each shape class per distinct shape."""
    import bench
    from newton_schulz_nesterov_gb300 import workloads
    sample, desc = bench.oracle_sample("llama3_8b")
    w = workloads.get("llama3_8b")
    shapes = {w.shapes[i]: (cnt, timed) for i, cnt, timed in sample}
    assert shapes == {(4096, 4096): (64, True), (1024, 4096): (64, True), (14336, 4096): (64, True),
                      (4096, 14336): (32, True)}
    assert sum(cnt for _, cnt, _ in sample) == len(w.shapes)
    big, _ = bench.oracle_sample("tp_70b_mixed")      # the 28672 x 8192 matrix is over the host budget
    assert [t for _, _, t in big] == [False, True]
