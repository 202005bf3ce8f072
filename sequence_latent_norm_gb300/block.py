"""The full MLA attention block around the per-rank LAGA compute.

Algorithm 1 of the LAGA page ("A Training-Memory Regression in MLA Sequence
Parallelism ... LAGA", Section 3.3), on one rank of P:

  step 1     q = h W_q and [latent | k_pe] = h W_kv_a on the rank's chunk
             of the sequence (the latent norm is applied by the compute,
             after the gather: it is per token, so the result is the same)
  steps 2-6  ``attn``: ``sp.SequenceParallelLaga`` (the q / O all-to-alls
             and the latent all-gather around laga_fwd), or, at one rank
             without a process group, the library directly
  step 7     y = reshape(out) W_o on the rank's chunk

W_q, W_kv_a and W_o are plain bias-free dense GEMMs: they run as torch
matmuls (cuBLAS on the GPU, in the I/O dtype with fp32 accumulation).
Every step of the LAGA compute itself runs in the library's kernels.

Backward, for the loss sum(y * dy):
  dW_o = out^T dy,  d_out = dy W_o^T,
  (dq, dc, dW_kv_b, dgamma) = attn.backward(d_out),
  dW_q = h^T dq,  dW_kv_a = h^T dc,  dh = dq W_q^T + dc W_kv_a^T.
Every rank holds the same W_q, W_kv_a and W_o and a different chunk of the
sequence, so their gradients are summed over the ranks (all-reduce);
``attn`` already assembles dW_kv_b along the head axis and sums dgamma.
The weight gradients come out of the GEMMs in the I/O dtype and are
returned in (at least) fp32.
"""

from __future__ import annotations

import collections

import torch.distributed as dist

from .sp import LibraryCompute, SequenceParallelLaga
from .api import Shard


def _wide(t):
    """A weight gradient in at least fp32."""
    return t.float() if t.element_size() < 4 else t


class LagaAttentionBlock:
    """One rank's attention block.  ``attn`` runs steps 2-6 (``forward(q,
    c, w_kvb, gamma, cos, sin) -> (out, lse)`` on the rank's chunk,
    ``backward(d_out) -> (dq, dc, dw_kvb, dgamma)``); ``group`` is the
    process group whose ranks share the weights (None: one rank, no
    collective)."""

    def __init__(self, attn, n_h: int, group=None, distributed: bool = False):
        self.attn = attn
        self.n_h = n_h
        self.group = group
        self.distributed = distributed
        self.sent = collections.Counter()
        self._saved = None

    @classmethod
    def sequence_parallel(cls, n_h: int, S: int, *, group=None, device=None, **dims):
        """A rank of a sequence-parallel group (torch.distributed must be
        initialised): the library on its n_h/P heads behind sp.py's
        exchanges."""
        return cls(SequenceParallelLaga(n_h, S, group=group, device=device, **dims), n_h, group,
                   distributed=True)

    @classmethod
    def single(cls, n_h: int, S: int, *, device=None, B: int = 1, **dims):
        """All n_h heads and the whole sequence on one device, no process
        group: the library directly."""
        shard = Shard(S=S, H=n_h, n_h_total=n_h, B=B, **dims)
        return cls(LibraryCompute(shard, device), n_h)

    def forward(self, h, w_q, w_kva, gamma, w_kvb, w_o, cos, sin):
        """h [B, S_r, d_model] (this rank's chunk); w_q [d_model, n_h (d_nope
        + d_rope)]; w_kva [d_model, d_kv + d_rope]; gamma [d_kv] fp32;
        w_kvb [d_kv, n_h (d_nope + d_v)]; w_o [n_h d_v, d_model]; cos/sin
        [S, d_rope/2] fp32 for the full sequence.  Returns y [B, S_r,
        d_model] in h's dtype."""
        B, S_r, d_model = h.shape
        h_flat = h.reshape(B * S_r, d_model)
        q = (h_flat @ w_q).reshape(B, S_r, self.n_h, -1)
        c = (h_flat @ w_kva).reshape(B, S_r, -1)
        out, _ = self.attn.forward(q, c, w_kvb, gamma, cos, sin)
        out_flat = out.reshape(B * S_r, -1)
        self._saved = (h_flat, w_q, w_kva, w_o, out_flat, out.shape, h.shape)
        return (out_flat @ w_o).reshape(B, S_r, d_model)

    def _all_reduce(self, t, what):
        if not self.distributed:
            return t
        P = dist.get_world_size(self.group)
        self.sent[what] += 2 * (P - 1) * t.numel() * t.element_size() // P
        dist.all_reduce(t, group=self.group)
        return t

    def backward(self, dy):
        """dy [B, S_r, d_model] (the rank's chunk).  Returns a dict: dh
        [B, S_r, d_model] in h's dtype; dw_q, dw_kva, dw_o (fp32, summed
        over the ranks); dw_kvb [d_kv, n_h (d_nope + d_v)] and dgamma
        [d_kv] (fp32, from ``attn``)."""
        h_flat, w_q, w_kva, w_o, out_flat, out_shape, h_shape = self._saved
        dy_flat = dy.reshape(h_flat.shape[0], -1)
        dw_o = _wide(out_flat.t() @ dy_flat)
        d_out = (dy_flat @ w_o.t()).reshape(out_shape)
        dq, dc, dw_kvb, dgamma = self.attn.backward(d_out)
        dq_flat = dq.reshape(h_flat.shape[0], -1)
        dc_flat = dc.reshape(h_flat.shape[0], -1).to(dq.dtype)
        dh = (dq_flat @ w_q.t() + dc_flat @ w_kva.t()).reshape(h_shape)
        dw_q = _wide(h_flat.t() @ dq_flat)
        dw_kva = _wide(h_flat.t() @ dc_flat)
        return dict(dh=dh, dw_q=self._all_reduce(dw_q, "all_reduce_dw_q"),
                    dw_kva=self._all_reduce(dw_kva, "all_reduce_dw_kva"),
                    dw_o=self._all_reduce(dw_o, "all_reduce_dw_o"),
                    dw_kvb=dw_kvb, dgamma=dgamma)
