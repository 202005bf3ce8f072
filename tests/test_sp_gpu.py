"""The sequence-parallel wrapper on the GPU with the library's compute: one
NCCL rank (every run here has one GPU), whose collectives reduce to local
copies, must give exactly what laga_fwd / laga_bwd give directly."""

import socket

import pytest
import torch
import torch.distributed as dist

from _harness import shard_of
from laga_inputs import config, make_inputs

pytestmark = pytest.mark.gpu


def test_single_rank_sequence_parallel_equals_direct_call():
    import sequence_latent_norm_gb300 as pkg
    from sequence_latent_norm_gb300.sp import SequenceParallelLaga
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        wl = config(1, S=640, H=4, n_h_total=4)
        t = {k: v.to(dev) for k, v in make_inputs(wl).items()}
        run = pkg.Laga(shard_of(wl), device=dev)
        o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
        ref = run.backward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"], o, lse, t["dO"])
        sp = SequenceParallelLaga(wl.n_h_total, wl.S, device=dev)
        o2, lse2 = sp.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
        got = sp.backward(t["dO"])
        pkg._lib.sync_check()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
        assert sp.sent["all_to_all_q"] == 0 and sp.sent["all_gather_c"] == 0
    finally:
        dist.destroy_process_group()
