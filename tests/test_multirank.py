"""The bench's multi-rank logic on CPU with real torch.distributed ranks (gloo, world size 2):
the layer shards over tokens with no exchange, so the only cross-rank steps are the barrier and
the max-over-ranks of the timings; the whole-job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank               # rank 1 is the slowest
        ms = bench.max_over_ranks(local_ms, "cpu")
        dist.barrier()
        tput = bench.job_tokens_per_s(world, 4096, 20, ms)
        q.put((rank, ms, tput, bench.runs_reference_arm(rank)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_take_the_slowest_time(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = 10.0 + 5.0 * (world - 1)
    for rank, ms, tput, ref in res:
        assert ms == slowest                        # every rank sees the max
        assert tput == pytest.approx(world * 4096 * 20 / (slowest / 1e3))
        assert ref == (rank == 0)                   # only rank 0 runs the reference arm


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(12.5, "cpu") == 12.5
    assert bench.job_tokens_per_s(1, 4096, 10, 20.0) == pytest.approx(4096 * 10 / 0.02)
