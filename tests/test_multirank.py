"""Multi-process (gloo, world_size 2) checks of the benchmark's rank logic:
the timed region takes the max over ranks and the value is the whole-job
(weak-scaling) throughput.  CPU only."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [1.0 + rank, 10.0 - rank]          # per-rank timings (s)
    got = bench.max_over_ranks(mine, dist)
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0]


def test_single_rank_and_weak_scaling():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.weak_scaling_value(100.0, 4, 2.0) == 200.0


def test_gemv_bytes_formula():
    import bench
    # N*K/2 packed + N*K/16 scales + 2*M*K activation + 2*M*N output + 4 (global scale)
    assert bench.gemv_bytes(4, 5120, 5120) == 5120 * 2560 + 5120 * 320 + 2 * 4 * 5120 * 2 + 4
    assert bench.dequant_bytes(17408, 5120) == 17408 * 2560 + 17408 * 320 + 2 * 17408 * 5120 + 4
