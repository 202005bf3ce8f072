"""Sequence-parallel LAGA across ranks: the collectives of Algorithm 1.

The LAGA page ("A Training-Memory Regression in MLA Sequence Parallelism
... LAGA", Section 3.3, Algorithm 1 and Section 5.2) runs one attention
layer over P ranks that each start with a contiguous chunk of the sequence
for all heads.  Per rank and step:

  forward   all-gather of the latent c = [latent | k_pe] over the sequence
            (step 3); all-to-all of q from sequence chunks to head shards
            (step 2); the rank's compute on its n_h/P heads over the full
            sequence (steps 4-5: latent norm, RoPE, up-projection, causal
            attention -- this library's laga_fwd); all-to-all of O back to
            sequence chunks (step 6).
  backward  all-to-all of dO to head shards; laga_bwd; all-to-all of dq
            back; reduce-scatter (sum) of the rank's partial dc to sequence
            chunks; the W_kv_b gradient, computed per head shard, assembled
            along the head axis; all-reduce (sum) of dgamma.

The latent norm is a per-token operation, so applying it after the gather
(inside laga_fwd, as here) gives the same result as before it.  Every
collective goes through torch.distributed on the group's tensors: with
NCCL on GPUs the gathered latent lands in local HBM before the compute
reads it.  Backends without all-to-all (gloo) exchange the chunks
point to point instead, with the same payload.

``SequenceParallelLaga`` counts the bytes each collective of one step
sends from this rank (``sent``), and the element counts that the page's
communication accounting (Section 4.2, Table 1) is stated in
(``forward_elements``).
"""

from __future__ import annotations

import collections

import torch
import torch.distributed as dist

from .api import Laga, Shard


class LibraryCompute:
    """The per-rank compute of one head shard on the GPU: laga_fwd and
    laga_bwd of this library (the default compute of SequenceParallelLaga)."""

    def __init__(self, shard: Shard, device):
        self.run = Laga(shard, device=device)
        self.saved = None

    def forward(self, q, c, w, gamma, cos, sin):
        o, lse = self.run.forward(q, c, w, gamma, cos, sin)
        self.saved = (q, c, w, gamma, cos, sin, o, lse)
        return o, lse

    def backward(self, d_o):
        q, c, w, gamma, cos, sin, o, lse = self.saved
        return self.run.backward(q, c, w, gamma, cos, sin, o, lse, d_o)


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


class SequenceParallelLaga:
    """One rank of sequence-parallel LAGA over ``group``.

    n_h heads, full sequence S (a multiple of P); the rank computes heads
    [rank * n_h/P, (rank + 1) * n_h/P).  ``compute`` runs one head shard
    (``forward(q, c, w, gamma, cos, sin) -> (O, LSE)``, ``backward(dO) ->
    (dq, dc, dw, dgamma)``); by default it is this library on ``device``.
    """

    def __init__(self, n_h: int, S: int, *, group=None, B: int = 1, d_nope: int = 128,
                 d_rope: int = 64, d_v: int = 128, d_kv: int = 512, io_dtype: str = "bf16",
                 norm: str = "layer", device=None, compute=None):
        self.group = group
        self.P = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if n_h % self.P or S % self.P:
            raise ValueError(f"n_h={n_h} and S={S} must be multiples of the {self.P} ranks")
        self.n_h, self.S, self.B = n_h, S, B
        self.H = n_h // self.P
        self.Sr = S // self.P
        self.dims = dict(d_nope=d_nope, d_rope=d_rope, d_v=d_v, d_kv=d_kv)
        if compute is None:
            shard = Shard(S=S, H=self.H, n_h_total=n_h, head_offset=self.rank * self.H, B=B,
                          io_dtype=io_dtype, norm=norm, **self.dims)
            compute = LibraryCompute(shard, device)
        self.compute = compute
        self.sent = collections.Counter()
        self._a2a_native = dist.get_backend(group) != "gloo"

    # ------------------------------------------------------------ collectives
    def _all_to_all(self, outs, ins, what):
        """outs[p] <- rank p's ins[self.rank]; counts the off-rank payload."""
        self.sent[what] += sum(_nbytes(t) for p, t in enumerate(ins) if p != self.rank)
        if self._a2a_native:
            dist.all_to_all(outs, ins, group=self.group)
            return
        reqs = []
        for p in range(self.P):
            if p == self.rank:
                outs[p].copy_(ins[p])
                continue
            peer = dist.get_global_rank(self.group, p) if self.group is not None else p
            reqs.append(dist.isend(ins[p].contiguous(), peer, group=self.group))
            reqs.append(dist.irecv(outs[p], peer, group=self.group))
        for r in reqs:
            r.wait()

    def _heads_from_seq(self, x_local, what):
        """[B, S/P, n_h, d] sequence chunk -> [B, S, n_h/P, d] head shard."""
        ins = [x_local[:, :, p * self.H:(p + 1) * self.H].contiguous() for p in range(self.P)]
        outs = [torch.empty_like(ins[0]) for _ in range(self.P)]
        self._all_to_all(outs, ins, what)
        return torch.cat(outs, dim=1)

    def _seq_from_heads(self, x_mine, what):
        """[B, S, n_h/P, d] head shard -> [B, S/P, n_h, d] sequence chunk."""
        ins = [x_mine[:, p * self.Sr:(p + 1) * self.Sr].contiguous() for p in range(self.P)]
        outs = [torch.empty_like(ins[0]) for _ in range(self.P)]
        self._all_to_all(outs, ins, what)
        return torch.cat(outs, dim=2)

    # ------------------------------------------------------------ passes
    def forward(self, q_local, c_local, w, gamma, cos, sin):
        """q_local [B, S/P, n_h, d_nope + d_rope] and c_local [B, S/P,
        d_kv + d_rope]: this rank's sequence chunk; w [d_kv, n_h (d_nope +
        d_v)], gamma [d_kv] and cos/sin [S, d_rope/2] (full sequence) as for
        laga_fwd.  Returns O [B, S/P, n_h, d_v] for the rank's chunk and the
        LSE [B, n_h/P, S] of its heads."""
        self.sent.clear()
        chunks = [torch.empty_like(c_local) for _ in range(self.P)]
        self.sent["all_gather_c"] += (self.P - 1) * _nbytes(c_local)
        dist.all_gather(chunks, c_local.contiguous(), group=self.group)
        c_full = torch.cat(chunks, dim=1)
        q_mine = self._heads_from_seq(q_local, "all_to_all_q")
        o_mine, lse = self.compute.forward(q_mine, c_full, w, gamma, cos, sin)
        self._elems = dict(q=q_local.numel(), o=o_mine.numel(), c=c_local.numel())
        return self._seq_from_heads(o_mine, "all_to_all_o"), lse

    def backward(self, d_o_local):
        """dO [B, S/P, n_h, d_v] of the rank's chunk.  Returns dq [B, S/P,
        n_h, d_nope + d_rope] and dc [B, S/P, d_kv + d_rope] of the chunk
        (summed over all ranks' heads), the full W_kv_b gradient [d_kv,
        n_h (d_nope + d_v)] and dgamma [d_kv], summed over ranks."""
        d_o_mine = self._heads_from_seq(d_o_local, "all_to_all_do")
        dq_mine, dc_part, dw_mine, dg_part = self.compute.backward(d_o_mine)
        dq_local = self._seq_from_heads(dq_mine, "all_to_all_dq")
        dc_chunks = [dc_part[:, p * self.Sr:(p + 1) * self.Sr].contiguous()
                     for p in range(self.P)]
        dc_local = torch.empty_like(dc_chunks[0])
        self.sent["reduce_scatter_dc"] += sum(_nbytes(t) for p, t in enumerate(dc_chunks)
                                              if p != self.rank)
        dist.reduce_scatter(dc_local, dc_chunks, group=self.group)
        cols = [torch.empty_like(dw_mine) for _ in range(self.P)]
        self.sent["all_gather_dw"] += (self.P - 1) * _nbytes(dw_mine)
        dist.all_gather(cols, dw_mine.contiguous(), group=self.group)
        dw = torch.cat(cols, dim=1)
        dgamma = dg_part.clone()
        self.sent["all_reduce_dgamma"] += 2 * (self.P - 1) * _nbytes(dgamma) // self.P
        dist.all_reduce(dgamma, group=self.group)
        return dq_local, dc_local, dw, dgamma

    def forward_elements(self):
        """Elements this rank moves in the forward, in the terms of the
        page's accounting (Section 4.2, Table 1): the off-rank part of the q
        and O all-to-alls, and its own chunk of the gathered latent."""
        off = (self.P - 1) / self.P
        return dict(q=off * self._elems["q"], o=off * self._elems["o"], latent=self._elems["c"])
