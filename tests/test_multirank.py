"""The N > 1 launch path of the benchmark on CPU: two gloo ranks run the timing
helpers a multi-GPU run uses (rank discovery from the launcher's environment,
barrier, max over ranks, whole-job aggregate), and the reference arm's rank
filter.  The path shards by sequence (replicas, no data-path collective), so these
helpers are all the N > 1 run adds."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="env://")
    try:
        w, r, lr = bench.dist_setup()
        assert (w, r, lr) == (world, rank, rank)
        # each rank "times" its own replica: rank r took 1 + r seconds for 10 units
        secs = bench.max_over_ranks(1.0 + rank, world)
        assert secs == float(world)  # the slowest rank sets the job's time
        bench.barrier(world)
        value = bench.aggregate(10.0, secs, world)
        assert value == 10.0 * world / world
        # the reference arm prints on rank 0 only
        args = type("A", (), {"seed": 0, "warmup": 3, "steps": 1, "cpu_budget": 0.01})()
        if rank != 0:
            assert bench.run_reference(args) is None
        with open(os.path.join(out_dir, f"ok{rank}"), "w") as f:
            f.write(f"{secs} {value}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    ctx = mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                             join=True, start_method="spawn")
    del ctx
    for r in range(world):
        assert (tmp_path / f"ok{r}").read_text() == "2.0 10.0"
