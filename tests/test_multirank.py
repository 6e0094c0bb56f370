"""The benchmark's multi-rank path on the CPU with gloo (world size 2): every rank runs its own
replica of the workload; the ranks only meet in the max-reduction of their timings."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import gdr_inputs as gi
    # per-rank timings: the reduction must return the slowest rank's value element-wise
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0], "cpu", world)
    # each rank draws a different replica of the same workload (seed offset = rank)
    wl = gi.custom(seqlens=[16], H=1, d_k=8, d_v=8, dtype="f32")
    x = gi.device_full(wl, "cpu", seed_offset=rank)["q"]
    xs = [torch.zeros_like(x) for _ in range(world)]
    dist.all_gather(xs, x)
    dist.barrier()
    q.put((rank, got, bool(torch.equal(xs[0], xs[1]))))
    dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for rank, got, same in res:
        assert got == [2.0, 10.0, 3.0]
        assert not same  # replicas hold different synthetic inputs


def test_job_throughput():
    import bench
    assert bench.job_tokens_per_s(4, 1000, 0.5) == pytest.approx(8000.0)
