"""Sequence-parallel LAGA on CPU ranks (gloo): the collectives of Algorithm 1
around a per-rank compute, checked against the unsharded fp64 oracle, and
the bytes each rank sends checked against the page's accounting
(Section 4.2, Table 1).

Each rank starts from its sequence chunk of q and c for all heads; the
per-rank compute here is the oracle's forward/backward of the rank's head
shard (the GPU compute is the library, tested on the GPU), so these tests
cover the exchange: the latent all-gather, the q/O/dO/dq all-to-alls, the
dc reduce-scatter, the head-axis assembly of dW_kv_b and the dgamma
all-reduce.
"""

import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


class OracleCompute:
    """The per-rank compute of one head shard, by the fp64 oracle."""

    def __init__(self, dims):
        self.dims = dims

    def forward(self, q, c, w, gamma, cos, sin):
        O, LSE, self.st = oracle.forward(q.numpy(), c.numpy(), w.numpy(), gamma.numpy(),
                                         cos.numpy(), sin.numpy(), self.dims)
        return torch.from_numpy(O), torch.from_numpy(LSE)

    def backward(self, d_o):
        g = oracle.backward(self.st, d_o.numpy())
        return tuple(torch.from_numpy(np.ascontiguousarray(g[k]))
                     for k in ("dq", "dc", "dw", "dgamma"))


def _problem(n_h, S, dims, seed=7):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, S, n_h, dims["d_nope"] + dims["d_rope"]))
    c = rng.standard_normal((1, S, dims["d_kv"] + dims["d_rope"]))
    w = rng.standard_normal((dims["d_kv"], n_h * (dims["d_nope"] + dims["d_v"]))) / \
        math.sqrt(dims["d_kv"])
    gamma = 1.0 + 0.1 * rng.standard_normal(dims["d_kv"])
    cos, sin = oracle.rope_tables(S, dims["d_rope"])
    d_o = rng.standard_normal((1, S, n_h, dims["d_v"]))
    return q, c, w, gamma, cos, sin, d_o


def _rank(rank, world, port, n_h, S, dims, norm):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sequence_latent_norm_gb300.sp import SequenceParallelLaga
        q, c, w, gamma, cos, sin, d_o = _problem(n_h, S, dims)
        full = oracle.Dims(S=S, H=n_h, norm=norm, **dims)
        O, LSE, st = oracle.forward(q, c, w, gamma, cos, sin, full)
        g = oracle.backward(st, d_o)
        P, H, Sr = world, n_h // world, S // world
        mine = oracle.Dims(S=S, H=H, n_h_total=n_h, head_offset=rank * H, norm=norm, **dims)
        sp = SequenceParallelLaga(n_h, S, compute=OracleCompute(mine), norm=norm, **dims)
        seq = slice(rank * Sr, (rank + 1) * Sr)
        T = torch.from_numpy
        o_loc, lse = sp.forward(T(q[:, seq]).contiguous(), T(c[:, seq]).contiguous(), T(w),
                                T(gamma), T(cos), T(sin))
        fwd_sent = dict(sp.sent)
        elems = sp.forward_elements()
        dq, dc, dw, dg = sp.backward(T(d_o[:, seq]).contiguous())
        tol = dict(rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(o_loc.numpy(), O[:, seq], **tol)
        np.testing.assert_allclose(lse.numpy(), LSE[:, rank * H:(rank + 1) * H], **tol)
        np.testing.assert_allclose(dq.numpy(), g["dq"][:, seq], **tol)
        np.testing.assert_allclose(dc.numpy(), g["dc"][:, seq], **tol)
        np.testing.assert_allclose(dw.numpy(), g["dw"], **tol)
        np.testing.assert_allclose(dg.numpy(), g["dgamma"], **tol)
        # the page's accounting: 4-byte q and O elements over the all-to-alls
        # (off-rank part), the latent chunk at 2 bytes an element
        table = 4 * (elems["q"] + elems["o"]) + 2 * elems["latent"]
        ref = oracle.comm_bytes_per_rank("laga", S, P, n_h=n_h, **dims)
        assert abs(table - ref) <= 1e-9 * ref, (table, ref)
        # wire bytes this rank sent (fp64 elements here), per collective
        off = (P - 1) / P
        qk = dims["d_nope"] + dims["d_rope"]
        assert fwd_sent["all_to_all_q"] == off * Sr * n_h * qk * 8
        assert fwd_sent["all_to_all_o"] == off * Sr * n_h * dims["d_v"] * 8
        assert fwd_sent["all_gather_c"] == (P - 1) * Sr * (dims["d_kv"] + dims["d_rope"]) * 8
        assert sp.sent["reduce_scatter_dc"] == off * S * (dims["d_kv"] + dims["d_rope"]) * 8
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SMALL = dict(d_nope=8, d_rope=4, d_v=6, d_kv=12)


@pytest.mark.parametrize("world,n_h,S,norm", [(2, 4, 12, "layer"), (4, 8, 16, "layer"),
                                              (2, 2, 10, "rms")])
def test_sequence_parallel_laga_matches_unsharded_oracle(world, n_h, S, norm):
    mp.spawn(_rank, args=(world, _free_port(), n_h, S, SMALL, norm), nprocs=world, join=True)


def test_sequence_parallel_comm_at_deepseek_v3_dims_matches_table1_form():
    """DeepSeek-V3 dims (d_nope = d_v = 128, d_rope = 64, d_kv = 512), 2
    ranks, one head each over a short sequence: the per-rank forward bytes
    in the page's accounting equal the closed form that reproduces Table 1
    (which is linear in S, so equality here is equality at S = 4K-16K)."""
    dims = dict(d_nope=128, d_rope=64, d_v=128, d_kv=512)
    mp.spawn(_rank, args=(2, _free_port(), 2, 8, dims, "layer"), nprocs=2, join=True)


def _rank_block(rank, world, port, n_h, S, dims, d_model):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle.block import block_backward, block_forward
        from sequence_latent_norm_gb300.block import LagaAttentionBlock
        from sequence_latent_norm_gb300.sp import SequenceParallelLaga
        rng = np.random.default_rng(11)
        qk, hkv = dims["d_nope"] + dims["d_rope"], dims["d_nope"] + dims["d_v"]
        h = rng.standard_normal((1, S, d_model))
        w_q = rng.standard_normal((d_model, n_h * qk)) / math.sqrt(d_model)
        w_kva = rng.standard_normal((d_model, dims["d_kv"] + dims["d_rope"])) / math.sqrt(d_model)
        gamma = 1.0 + 0.1 * rng.standard_normal(dims["d_kv"])
        w_kvb = rng.standard_normal((dims["d_kv"], n_h * hkv)) / math.sqrt(dims["d_kv"])
        w_o = rng.standard_normal((n_h * dims["d_v"], d_model)) / math.sqrt(n_h * dims["d_v"])
        cos, sin = oracle.rope_tables(S, dims["d_rope"])
        dy = rng.standard_normal((1, S, d_model))
        full = oracle.Dims(S=S, H=n_h, **dims)
        y, st = block_forward(h, w_q, w_kva, gamma, w_kvb, w_o, cos, sin, full)
        g = block_backward(st, dy)
        P, H, Sr = world, n_h // world, S // world
        mine = oracle.Dims(S=S, H=H, n_h_total=n_h, head_offset=rank * H, **dims)
        sp = SequenceParallelLaga(n_h, S, compute=OracleCompute(mine), **dims)
        blk = LagaAttentionBlock(sp, n_h, distributed=True)
        seq = slice(rank * Sr, (rank + 1) * Sr)
        T = torch.from_numpy
        y_loc = blk.forward(T(h[:, seq]).contiguous(), T(w_q), T(w_kva), T(gamma), T(w_kvb),
                            T(w_o), T(cos), T(sin))
        got = blk.backward(T(dy[:, seq]).contiguous())
        tol = dict(rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(y_loc.numpy(), y[:, seq], **tol)
        np.testing.assert_allclose(got["dh"].numpy(), g["dh"][:, seq], **tol)
        for k in ("dw_q", "dw_kva", "dw_o", "dw_kvb", "dgamma"):
            np.testing.assert_allclose(got[k].numpy(), g[k], **tol, err_msg=k)
        # the three replicated weights' gradients are all-reduced: ring bytes
        # 2 (P-1)/P of each fp64 gradient
        for k, w in (("dw_q", w_q), ("dw_kva", w_kva), ("dw_o", w_o)):
            assert blk.sent["all_reduce_" + k] == 2 * (P - 1) * w.size * 8 // P
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n_h,S", [(2, 4, 12), (4, 4, 8)])
def test_sequence_parallel_attention_block_matches_unsharded_block_oracle(world, n_h, S):
    """The whole block of Algorithm 1 (W_q, W_kv_a, the exchanges around the
    per-rank compute, W_o) on CPU ranks equals the unsharded block oracle:
    y and dh per sequence chunk, and the summed weight gradients."""
    mp.spawn(_rank_block, args=(world, _free_port(), n_h, S, SMALL, 7), nprocs=world, join=True)
