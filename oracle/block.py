"""Plain fp64 oracle of the full MLA attention block around the LAGA compute.

TEST INFRASTRUCTURE ONLY (see the package docstring): used by ``tests/`` and
nowhere in the product path.

The block is Algorithm 1 of the LAGA page ("A Training-Memory Regression in
MLA Sequence Parallelism ... LAGA", Section 3.3), written at one rank:

  step 1  q = h W_q, split per head into (q_nope | q_rope);
          [latent | k_pe] = h W_kv_a;  the latent norm is part of the
          per-rank compute (``forward``), where the method applies it
  steps 2, 3, 6  the head / sequence exchanges, identities at one rank
                 (their sharded form is checked against this unsharded
                 result by the sequence-parallel tests)
  steps 4-5  ``forward`` of this package: norm, RoPE, up-projection,
             causal attention
  step 7  y = reshape(out) W_o

Readings where the page leaves the block open: W_q, W_kv_a and W_o are
plain bias-free linear maps (the algorithm writes them as such; the
DeepSeek-V3 query low-rank path is not on the page), and the output keeps
the head-major column order of reshape(out) = [out_head0 | out_head1 | ...].

Backward, for the loss sum(y * dy), by the chain rule through the three
linear maps around ``backward``:
  dW_o = out^T dy,   d_out = dy W_o^T,
  (dq, dc, dW_kv_b, dgamma) = backward(d_out),
  dW_q = h^T dq,   dW_kv_a = h^T dc,   dh = dq W_q^T + dc W_kv_a^T.

Parity status: pinned by central finite differences of ``block_forward``
in every input and weight (tests/test_oracle_block.py) and by the identity
with ``forward`` / ``backward`` when the projections are the identity.
"""

from __future__ import annotations

import numpy as np

from .laga import Dims, backward, forward


def block_forward(h, w_q, w_kva, gamma, w_kvb, w_o, cos, sin, dims: Dims):
    """h [B, S, d_model]; w_q [d_model, n_h (d_nope + d_rope)];
    w_kva [d_model, d_kv + d_rope]; gamma [d_kv]; w_kvb [d_kv, n_h (d_nope +
    d_v)]; w_o [n_h d_v, d_model]; cos/sin [S, d_rope/2].  ``dims`` has
    H = n_h_total = n_h (all heads at one rank).  Returns (y [B, S, d_model],
    saved state for ``block_backward``)."""
    B, S, _ = h.shape
    n_h = dims.H
    q = (h @ w_q).reshape(B, S, n_h, dims.d_nope + dims.d_rope)
    c = h @ w_kva
    out, lse, st = forward(q, c, w_kvb, gamma, cos, sin, dims)
    y = out.reshape(B, S, n_h * dims.d_v) @ w_o
    return y, dict(h=h, w_q=w_q, w_kva=w_kva, w_o=w_o, out=out, lse=lse, attn=st)


def block_backward(saved, dy):
    """Gradients of sum(y * dy): dict with dh, dw_q, dw_kva, dgamma, dw_kvb,
    dw_o (shapes of the corresponding inputs)."""
    h, w_q, w_kva, w_o, out = (saved[k] for k in ("h", "w_q", "w_kva", "w_o", "out"))
    B, S, d_model = h.shape
    out_flat = out.reshape(B * S, -1)
    dy_flat = dy.reshape(B * S, d_model)
    dw_o = out_flat.T @ dy_flat
    d_out = (dy_flat @ w_o.T).reshape(out.shape)
    g = backward(saved["attn"], d_out)
    dq_flat = g["dq"].reshape(B * S, -1)
    dc_flat = g["dc"].reshape(B * S, -1)
    h_flat = h.reshape(B * S, d_model)
    dh = (dq_flat @ w_q.T + dc_flat @ w_kva.T).reshape(B, S, d_model)
    return dict(dh=dh, dw_q=h_flat.T @ dq_flat, dw_kva=h_flat.T @ dc_flat,
                dgamma=g["dgamma"], dw_kvb=g["dw"], dw_o=dw_o)


def block_flops(S, n_h, d_model, B=1, d_nope=128, d_rope=64, d_v=128, d_kv=512):
    """FLOPs of the block's three projections, forward and backward (2 GEMMs
    of the same size per weight in the backward), for B*S tokens."""
    T = B * S
    per = 2.0 * T * d_model * (n_h * (d_nope + d_rope) + (d_kv + d_rope) + n_h * d_v)
    return per, 2 * per


__all__ = ["block_forward", "block_backward", "block_flops"]
