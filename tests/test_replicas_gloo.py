"""The N-replica path of the benchmark on CPU: two gloo ranks, each with its
own timing; the whole-job rate uses the slowest rank, and the reference arm
runs on rank 0 alone."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_path):
    import sys

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    local_ms = 100.0 + 50.0 * rank            # rank 1 is the slow one
    value, slowest = bench.job_throughput(tokens_per_step=29, steps=10, elapsed_ms=local_ms,
                                          world=w)

    class Args:
        steps, warmup, gpus = 1, 0, world

    def no_reference_work(*args):
        raise RuntimeError("the reference arm works on rank 0 only")

    bench.host_layer_bits = no_reference_work
    if rank != 0:
        bench.run_reference(Args, None, w, r)   # returns at once: no work, no output
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(f"{value} {slowest}")
    dist.destroy_process_group()


def test_two_replicas_use_the_slowest_rank(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    out = str(tmp_path / "rank")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        value, slowest = open(f"{out}.{rank}").read().split()
        assert float(slowest) == 150.0
        assert float(value) == pytest.approx(29 * 10 * 2 / 0.150)
