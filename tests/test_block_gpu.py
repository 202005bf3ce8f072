"""The full attention block (W_q, W_kv_a, the library's LAGA compute, W_o)
on the GPU against the fp64 block oracle on the same bf16 inputs, and the
one-rank sequence-parallel block against the direct one."""

import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from _harness import RECORDS
from laga_inputs import as_f64, config, make_block_inputs

pytestmark = pytest.mark.gpu

# The block's outputs and weight gradients pass through bf16 storage at
# every GEMM boundary (q, c, out, d_out, dq, dc and the weight gradients
# themselves are bf16), each adding ~2^-9 relative rounding on top of the
# per-rank compute's own 1e-2 gradient bound.
BLOCK_REL_FRO = 1e-2


def _rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _run_block(blk, t):
    y = blk.forward(t["h"], t["w_q"], t["w_kva"], t["gamma"], t["w_kvb"], t["w_o"], t["cos"],
                    t["sin"])
    g = blk.backward(t["dy"])
    return y, g


@pytest.mark.parametrize("form", ["laga", "laga_fused"])
@pytest.mark.parametrize("case", [dict(S=640, H=4, d_model=384), dict(S=257, H=2, B=2, d_model=256)],
                         ids=["S640-H4", "S257-B2"])
def test_attention_block_matches_block_oracle(case, form):
    import sequence_latent_norm_gb300 as pkg
    from oracle import Dims
    from oracle.block import block_backward, block_forward
    from sequence_latent_norm_gb300.block import LagaAttentionBlock
    case = dict(case)
    d_model = case.pop("d_model")
    wl = config(1, n_h_total=case["H"], **case)
    cpu = make_block_inputs(wl, d_model)
    dev = torch.device("cuda:0")
    t = {k: v.to(dev) for k, v in cpu.items()}
    blk = LagaAttentionBlock.single(wl.H, wl.S, B=wl.B, device=dev, form=form)
    y, g = _run_block(blk, t)
    pkg._lib.sync_check()
    a = {k: as_f64(v) for k, v in cpu.items()}
    dims = Dims(S=wl.S, H=wl.H, B=wl.B)
    y_ref, st = block_forward(a["h"], a["w_q"], a["w_kva"], a["gamma"], a["w_kvb"], a["w_o"],
                              a["cos"], a["sin"], dims)
    ref = block_backward(st, a["dy"])
    errs = {"y": _rel_fro(as_f64(y), y_ref)}
    for k in ("dh", "dw_q", "dw_kva", "dw_o", "dw_kvb", "dgamma"):
        errs[k] = _rel_fro(as_f64(g[k]), ref[k])
    RECORDS.append((f"block {form} S={wl.S} H={wl.H} B={wl.B} d_model={d_model}",
                    {"block": errs}))
    for k, e in errs.items():
        assert e <= BLOCK_REL_FRO, f"{k}: rel-fro {e:.3e}"


def test_single_rank_sequence_parallel_block_equals_direct_block():
    import sequence_latent_norm_gb300 as pkg
    from sequence_latent_norm_gb300.block import LagaAttentionBlock
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        wl = config(1, S=384, H=4, n_h_total=4)
        t = {k: v.to(dev) for k, v in make_block_inputs(wl, 256).items()}
        y1, g1 = _run_block(LagaAttentionBlock.single(wl.H, wl.S, device=dev), t)
        y2, g2 = _run_block(LagaAttentionBlock.sequence_parallel(wl.H, wl.S, device=dev), t)
        pkg._lib.sync_check()
        assert torch.equal(y1, y2)
        for k in g1:
            assert torch.equal(g1[k], g2[k]), k
    finally:
        dist.destroy_process_group()
