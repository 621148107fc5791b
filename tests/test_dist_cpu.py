"""The bench's multi-rank host logic on CPU: two gloo ranks (the layout
torchrun gives the bench on N GPUs) set up the process group, pass a barrier
and agree on the max-over-ranks time; whole-job throughput sums the ranks'
independent work (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(0.5 + rank, w)  # per-rank "elapsed seconds"
    work = 1e12  # each rank's independent problem
    job = work * w / t
    q.put((rank, t, job))
    import torch.distributed as dist

    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU/gloo layout test")
def test_two_gloo_ranks_max_time_and_weak_scaling():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t, job in res:
        assert t == 1.5                 # max over ranks, not the local time
        assert job == pytest.approx(2 * 1e12 / 1.5)
