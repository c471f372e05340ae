"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own replica.

Every (batch, head) chain is independent, so N GPUs run N replicas with no data
exchange; the only cross-rank steps are the barrier around the timed region and
the max over ranks of the per-step time. This runs those steps for real with the
gloo backend (world size 2) and checks the whole-job throughput formula.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    ms = bench.max_over_ranks(1.0 + rank, w)  # rank 1 is the slower one
    out[rank] = (ms, bench.replica_throughput(w, 1000, ms))
    import torch.distributed as dist

    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == out[1]
    ms, value = out[0]
    assert ms == 2.0
    assert value == pytest.approx(2 * 1000 / 2.0e-3)  # both ranks' tokens over the slowest rank's time
