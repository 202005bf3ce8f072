"""Host logic of bench.py's N>1 path on CPU: two gloo ranks."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from laga_inputs import config
        wl = bench.rank_workload(config(2), rank, world)
        slowest = bench.max_over_ranks(10.0 + rank, world)
        out.put((rank, wl.head_offset, wl.H, wl.n_h_total, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_heads_and_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    offsets = [r[1] for r in res]
    assert offsets == [0, 16] and all(r[2] == 16 and r[3] == 32 for r in res)
    assert all(r[4] == 11.0 for r in res)          # max over ranks, seen by both
