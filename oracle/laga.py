"""fp64 NumPy oracle of the per-rank LAGA compute (test infrastructure only).

Source: "A Training-Memory Regression in MLA Sequence Parallelism: Why
Megatron-Core Forbids Absorption, and LAGA -- a Communication-Efficient Fix"
(arXiv 2607.17644v1).  Section references below are to that page.

Readings taken where the page is silent or garbled:

* Section 2.1 prints the key of the score as (q_nope || k_pe) with q in both
  factors; Algorithm 1 step 5 and the Section 5.1 equation make it
  (k_nope || k_pe).  That is used.
* The divisor sqrt(d) is sqrt(d_nope + d_rope), the per-head q/k width.
* "LN" is LayerNorm over the d_kv latent columns only: mean-subtracted,
  biased variance, gain gamma, no bias, eps = 1e-5.  k_pe is never
  normalised (Section 5.3: the band is never compressed).
* c is laid out [latent (d_kv) | k_pe (d_rope)].
* W_kv_b is [d_kv, n_h * (d_nope + d_v)]; the columns of head i are
  [k_nope (d_nope) | v (d_v)], and a head shard is a contiguous column slice.
* RoPE pairs element i with element i + d_rope/2 ("rotate half"), angle =
  pos * theta^(-2i/d_rope), positions 0..S-1 of the gathered sequence; it
  is applied to q_rope and to k_pe (the raw inputs); dq and dc are with
  respect to the raw inputs.
* Attention is causal: key j is visible to query i iff j <= i.
* LSE is the natural-log log-sum-exp of the scaled scores of each row.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

F64 = np.float64


@dataclasses.dataclass(frozen=True)
class Dims:
    """Problem sizes of one rank's head shard (Section 2.1 notation)."""

    S: int
    H: int  # heads in this shard (n_h / SP)
    d_nope: int = 128
    d_rope: int = 64
    d_v: int = 128
    d_kv: int = 512
    B: int = 1
    n_h_total: int | None = None  # columns of W_kv_b are n_h_total*(d_nope+d_v)
    head_offset: int = 0
    eps: float = 1e-5
    scale: float | None = None  # None -> 1/sqrt(d_nope + d_rope)
    norm: str = "layer"         # "layer": the page's LN; "rms": its RMS variant

    @property
    def d_qk(self) -> int:
        return self.d_nope + self.d_rope

    @property
    def d_head_kv(self) -> int:
        return self.d_nope + self.d_v

    @property
    def sm_scale(self) -> float:
        return (1.0 / math.sqrt(self.d_qk)) if self.scale is None else float(self.scale)

    @property
    def n_total(self) -> int:
        return self.H if self.n_h_total is None else self.n_h_total


# --------------------------------------------------------------------------
# Latent norm (Section 2.1 "kv = W_kv_b LN(latent)"; Algorithm 1 step 1)
# --------------------------------------------------------------------------
def layernorm(x, gamma, eps=1e-5):
    """LayerNorm over the last axis with gain only.

    Returns (L, mean, rstd, xhat) with xhat = (x - mean) * rstd and
    L = xhat * gamma; the variance is the biased (population) one.
    """
    x = np.asarray(x, F64)
    mean = x.mean(axis=-1)
    var = ((x - mean[..., None]) ** 2).mean(axis=-1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mean[..., None]) * rstd[..., None]
    return xhat * np.asarray(gamma, F64), mean, rstd, xhat


def rmsnorm(x, gamma, eps=1e-5):
    """RMS variant of the latent norm (an extension; the page's norm is LN):
    no mean subtraction, rstd = 1/sqrt(mean(x^2) + eps).

    Returns (L, mean, rstd, xhat) like ``layernorm``, with mean = 0 and
    xhat = x * rstd, L = xhat * gamma.
    """
    x = np.asarray(x, F64)
    rstd = 1.0 / np.sqrt((x * x).mean(axis=-1) + eps)
    xhat = x * rstd[..., None]
    return xhat * np.asarray(gamma, F64), np.zeros_like(rstd), rstd, xhat


def rmsnorm_backward(dL, xhat, rstd, gamma):
    """Gradient of L = xhat * gamma, xhat = x * rstd, with respect to x and
    gamma.  With g = dL * gamma and n features:
    dx = rstd * (g - xhat * mean(g * xhat)),
    dgamma = sum over all tokens of dL * xhat.
    """
    g = dL * np.asarray(gamma, F64)
    m2 = (g * xhat).mean(axis=-1, keepdims=True)
    dx = rstd[..., None] * (g - xhat * m2)
    dgamma = (dL * xhat).reshape(-1, dL.shape[-1]).sum(axis=0)
    return dx, dgamma


def latent_norm(x, gamma, dims):
    """The latent norm of step a1 that ``dims.norm`` selects."""
    return (rmsnorm if dims.norm == "rms" else layernorm)(x, gamma, dims.eps)


def latent_norm_backward(dL, xhat, rstd, gamma, dims):
    """Backward of ``latent_norm``."""
    return (rmsnorm_backward if dims.norm == "rms" else layernorm_backward)(dL, xhat, rstd, gamma)


def layernorm_backward(dL, xhat, rstd, gamma):
    """Gradient of L = xhat * gamma with respect to x and gamma.

    With g = dL * gamma and n features:
    dx = rstd * (g - mean(g) - xhat * mean(g * xhat)),
    dgamma = sum over all tokens of dL * xhat.
    """
    g = dL * np.asarray(gamma, F64)
    m1 = g.mean(axis=-1, keepdims=True)
    m2 = (g * xhat).mean(axis=-1, keepdims=True)
    dx = rstd[..., None] * (g - m1 - xhat * m2)
    dgamma = (dL * xhat).reshape(-1, dL.shape[-1]).sum(axis=0)
    return dx, dgamma


# --------------------------------------------------------------------------
# Decoupled RoPE band (Section 2.1 property P2, Section 5.3)
# --------------------------------------------------------------------------
def rope_tables(S, d_rope, theta=10000.0, pos0=0):
    """cos/sin tables [S, d_rope/2] for absolute positions pos0..pos0+S-1."""
    half = d_rope // 2
    i = np.arange(half, dtype=F64)
    inv_freq = theta ** (-2.0 * i / d_rope)
    pos = np.arange(pos0, pos0 + S, dtype=F64)
    ang = pos[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def _bcast_tables(x, cos, sin, seq_axis):
    shape = [1] * x.ndim
    shape[seq_axis] = cos.shape[0]
    shape[-1] = cos.shape[1]
    return np.asarray(cos, F64).reshape(shape), np.asarray(sin, F64).reshape(shape)


def rope(x, cos, sin, seq_axis=1):
    """Rotate pairs (i, i + d/2) of the last axis by the table angle."""
    x = np.asarray(x, F64)
    half = x.shape[-1] // 2
    c, s = _bcast_tables(x, cos, sin, seq_axis)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_transpose(g, cos, sin, seq_axis=1):
    """Apply the transpose (inverse) rotation: the gradient through rope()."""
    g = np.asarray(g, F64)
    half = g.shape[-1] // 2
    c, s = _bcast_tables(g, cos, sin, seq_axis)
    g1, g2 = g[..., :half], g[..., half:]
    return np.concatenate([g1 * c + g2 * s, g2 * c - g1 * s], axis=-1)


# --------------------------------------------------------------------------
# Explicit-attention forward on the head shard (Algorithm 1 steps 4-5,
# Section 5.1 equation: k_nope[i,t] = W^k[i] L[t], v[i,t] = W^v[i] L[t])
# --------------------------------------------------------------------------
def shard_weights(w, dims: Dims):
    """This shard's columns of W_kv_b as [d_kv, H, d_nope + d_v]."""
    dh = dims.d_head_kv
    w = np.asarray(w, F64)
    assert w.shape == (dims.d_kv, dims.n_total * dh), w.shape
    cols = w[:, dims.head_offset * dh:(dims.head_offset + dims.H) * dh]
    return cols.reshape(dims.d_kv, dims.H, dh)


def _prologue(q, c, w, gamma, cos, sin, dims: Dims):
    q = np.asarray(q, F64)
    c = np.asarray(c, F64)
    B, S, H = dims.B, dims.S, dims.H
    assert q.shape == (B, S, H, dims.d_qk), q.shape
    assert c.shape == (B, S, dims.d_kv + dims.d_rope), c.shape
    x = c[..., :dims.d_kv]
    L, mean, rstd, xhat = latent_norm(x, gamma, dims)
    kpe_r = rope(c[..., dims.d_kv:], cos, sin)              # [B,S,d_rope]
    q_nope = q[..., :dims.d_nope]                            # [B,S,H,d_nope]
    q_rope_r = rope(q[..., dims.d_nope:], cos, sin)          # [B,S,H,d_rope]
    W = shard_weights(w, dims)                               # [d_kv,H,dh]
    return dict(q_nope=q_nope, q_rope_r=q_rope_r, L=L, mean=mean, rstd=rstd,
                xhat=xhat, kpe_r=kpe_r, W=W, gamma=np.asarray(gamma, F64),
                cos=np.asarray(cos, F64), sin=np.asarray(sin, F64))


def _causal_block_scores(qa, ka, qb, kb, r0, r1, sc):
    """Scaled scores of query rows r0..r1-1 against keys 0..r1-1, masked.

    qa.ka^T + qb.kb^T is the (q_nope || q_rope)(k_nope || k_pe)^T product
    written as the sum of its two column bands.
    """
    s = (qa @ ka[:r1].T + qb @ kb[:r1].T) * sc
    rows = np.arange(r0, r1)[:, None]
    cols = np.arange(r1)[None, :]
    s[cols > rows] = -np.inf
    return s


def forward(q, c, w, gamma, cos, sin, dims: Dims, heads=None, block=512):
    """O [B,S,H,d_v] and LSE [B,H,S] of explicit causal MLA attention.

    ``heads`` restricts the attention (not the up-projection) to a subset of
    the shard's heads; the others are left as NaN.  Returns (O, LSE, saved).
    """
    st = _prologue(q, c, w, gamma, cos, sin, dims)
    B, S, H = dims.B, dims.S, dims.H
    KV = np.einsum("bsk,khd->bshd", st["L"], st["W"], optimize=True)        # [B,S,H,dh]
    k_nope = KV[..., :dims.d_nope]
    v = KV[..., dims.d_nope:]
    O = np.full((B, S, H, dims.d_v), np.nan)
    LSE = np.full((B, H, S), np.nan)
    sc = dims.sm_scale
    hs = range(H) if heads is None else heads
    for b in range(B):
        for h in hs:
            for r0 in range(0, S, block):
                r1 = min(S, r0 + block)
                s = _causal_block_scores(st["q_nope"][b, r0:r1, h], k_nope[b, :, h],
                                         st["q_rope_r"][b, r0:r1, h], st["kpe_r"][b],
                                         r0, r1, sc)
                m = s.max(axis=1)
                p = np.exp(s - m[:, None])
                l = p.sum(axis=1)
                LSE[b, h, r0:r1] = m + np.log(l)
                O[b, r0:r1, h] = (p / l[:, None]) @ v[b, :r1, h]
    st.update(KV=KV, O=O, LSE=LSE, heads=None if heads is None else list(heads),
              dims=dims)
    return O, LSE, st


def backward(saved, dO, block=512):
    """Gradients of sum(O * dO) (Section 5.2; hand-derived).

    P_ij = exp(s_ij - LSE_i); delta_i = sum_d dO_id O_id;
    dP_ij = dO_i . v_j; dS_ij = P_ij (dP_ij - delta_i);
    dv_j = sum_i P_ij dO_i; dq_i = scale sum_j dS_ij k_j;
    dk_j = scale sum_i dS_ij q_i (k_pe summed over heads);
    dW_shard = L^T dKV; dL = sum_h dKV_h W_h^T; then LayerNorm and RoPE
    backward.  Returns a dict with dq, dc, dw (the shard's columns,
    [d_kv, H*(d_nope+d_v)]), dgamma and the intermediates dKV, dkpe_r, dL.
    dc and dgamma are None when the forward ran on a head subset.
    """
    dims: Dims = saved["dims"]
    B, S, H = dims.B, dims.S, dims.H
    dO = np.asarray(dO, F64)
    O, LSE, KV = saved["O"], saved["LSE"], saved["KV"]
    k_nope = KV[..., :dims.d_nope]
    v = KV[..., dims.d_nope:]
    qn, qr, kr = saved["q_nope"], saved["q_rope_r"], saved["kpe_r"]
    sc = dims.sm_scale
    delta = (dO * O).sum(axis=-1)                              # [B,S,H]
    dq_nope = np.full_like(qn, np.nan)
    dq_rope_r = np.full_like(qr, np.nan)
    dKV = np.full_like(KV, np.nan)
    dkpe_r_h = np.zeros((B, S, H, dims.d_rope))
    hs = range(H) if saved["heads"] is None else saved["heads"]
    for b in range(B):
        for h in hs:
            dk = np.zeros((S, dims.d_nope))
            dv = np.zeros((S, dims.d_v))
            for r0 in range(0, S, block):
                r1 = min(S, r0 + block)
                s = _causal_block_scores(qn[b, r0:r1, h], k_nope[b, :, h],
                                         qr[b, r0:r1, h], kr[b], r0, r1, sc)
                P = np.exp(s - LSE[b, h, r0:r1, None])
                dOb = dO[b, r0:r1, h]
                dP = dOb @ v[b, :r1, h].T
                dS = P * (dP - delta[b, r0:r1, h, None])
                dv[:r1] += P.T @ dOb
                dq_nope[b, r0:r1, h] = sc * (dS @ k_nope[b, :r1, h])
                dq_rope_r[b, r0:r1, h] = sc * (dS @ kr[b, :r1])
                dk[:r1] += sc * (dS.T @ qn[b, r0:r1, h])
                dkpe_r_h[b, :r1, h] += sc * (dS.T @ qr[b, r0:r1, h])
            dKV[b, :, h, :dims.d_nope] = dk
            dKV[b, :, h, dims.d_nope:] = dv
    dq = np.concatenate([dq_nope, rope_transpose(dq_rope_r, saved["cos"], saved["sin"])],
                        axis=-1)
    out = dict(dq=dq, dKV=dKV, delta=delta, dkpe_r_heads=dkpe_r_h)
    dW = np.einsum("bsk,bshd->khd", saved["L"], np.nan_to_num(dKV, nan=0.0), optimize=True)
    dW[:, [h for h in range(H) if h not in set(hs)], :] = np.nan
    out["dw"] = dW.reshape(dims.d_kv, H * dims.d_head_kv)
    if saved["heads"] is not None:
        out.update(dc=None, dgamma=None, dL=None)
        return out
    dL = np.einsum("bshd,khd->bsk", dKV, saved["W"], optimize=True)
    dx, dgamma = latent_norm_backward(dL, saved["xhat"], saved["rstd"], saved["gamma"], dims)
    dkpe_r = dkpe_r_h.sum(axis=2)
    dkpe = rope_transpose(dkpe_r, saved["cos"], saved["sin"])
    out.update(dc=np.concatenate([dx, dkpe], axis=-1), dgamma=dgamma, dL=dL,
               dkpe_r=dkpe_r)
    return out


# --------------------------------------------------------------------------
# Absorbed form B2 (Section 3.2; Figure 2): q_absorbed = W_kv_b^{k T} q_nope,
# attention in latent space, post-attention latent accumulator, V
# up-projection afterwards ("un-absorb").
# --------------------------------------------------------------------------
def forward_absorbed(q, c, w, gamma, cos, sin, dims: Dims, block=512):
    """Absorbed-form forward.  Returns (O, LSE, saved) like ``forward``.

    q_abs[b,s,h,:] = W^k[h] q_nope[b,s,h]            ([d_kv])
    s_ij = (q_abs_i . L_j + q_rope_i . k_pe_j) * scale
    o_lat_i = sum_j P_ij L_j                          ([d_kv])
    O_i = W^v[h]^T o_lat_i
    """
    st = _prologue(q, c, w, gamma, cos, sin, dims)
    B, S, H = dims.B, dims.S, dims.H
    Wk = st["W"][..., :dims.d_nope]                          # [d_kv,H,d_nope]
    Wv = st["W"][..., dims.d_nope:]                          # [d_kv,H,d_v]
    q_abs = np.einsum("bshd,khd->bshk", st["q_nope"], Wk, optimize=True)    # [B,S,H,d_kv]
    o_lat = np.zeros((B, S, H, dims.d_kv))
    LSE = np.zeros((B, H, S))
    sc = dims.sm_scale
    for b in range(B):
        for h in range(H):
            for r0 in range(0, S, block):
                r1 = min(S, r0 + block)
                s = _causal_block_scores(q_abs[b, r0:r1, h], st["L"][b],
                                         st["q_rope_r"][b, r0:r1, h], st["kpe_r"][b],
                                         r0, r1, sc)
                m = s.max(axis=1)
                p = np.exp(s - m[:, None])
                l = p.sum(axis=1)
                LSE[b, h, r0:r1] = m + np.log(l)
                o_lat[b, r0:r1, h] = (p / l[:, None]) @ st["L"][b, :r1]
    O = np.einsum("bshk,khd->bshd", o_lat, Wv, optimize=True)
    st.update(q_abs=q_abs, o_lat=o_lat, O=O, LSE=LSE, Wk=Wk, Wv=Wv, dims=dims)
    return O, LSE, st


def backward_absorbed(saved, dO, block=512):
    """Absorbed-form backward; same outputs as ``backward``."""
    dims: Dims = saved["dims"]
    B, S, H = dims.B, dims.S, dims.H
    dO = np.asarray(dO, F64)
    L, kr, qr = saved["L"], saved["kpe_r"], saved["q_rope_r"]
    q_abs, o_lat, LSE = saved["q_abs"], saved["o_lat"], saved["LSE"]
    sc = dims.sm_scale
    dWv = np.einsum("bshk,bshd->khd", o_lat, dO, optimize=True)
    do_lat = np.einsum("bshd,khd->bshk", dO, saved["Wv"], optimize=True)
    delta = (dO * saved["O"]).sum(axis=-1)
    dq_abs = np.zeros_like(q_abs)
    dq_rope_r = np.zeros_like(qr)
    dLat = np.zeros_like(L)
    dkpe_r = np.zeros_like(kr)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, S, block):
                r1 = min(S, r0 + block)
                s = _causal_block_scores(q_abs[b, r0:r1, h], L[b], qr[b, r0:r1, h], kr[b],
                                         r0, r1, sc)
                P = np.exp(s - LSE[b, h, r0:r1, None])
                dP = do_lat[b, r0:r1, h] @ L[b, :r1].T
                dS = P * (dP - delta[b, r0:r1, h, None])
                dq_abs[b, r0:r1, h] = sc * (dS @ L[b, :r1])
                dq_rope_r[b, r0:r1, h] = sc * (dS @ kr[b, :r1])
                dLat[b, :r1] += sc * (dS.T @ q_abs[b, r0:r1, h]) + P.T @ do_lat[b, r0:r1, h]
                dkpe_r[b, :r1] += sc * (dS.T @ qr[b, r0:r1, h])
    dWk = np.einsum("bshk,bshd->khd", dq_abs, saved["q_nope"], optimize=True)
    dq_nope = np.einsum("bshk,khd->bshd", dq_abs, saved["Wk"], optimize=True)
    dq = np.concatenate([dq_nope, rope_transpose(dq_rope_r, saved["cos"], saved["sin"])],
                        axis=-1)
    dW = np.concatenate([dWk, dWv], axis=-1).reshape(dims.d_kv, H * dims.d_head_kv)
    dx, dgamma = latent_norm_backward(dLat, saved["xhat"], saved["rstd"], saved["gamma"], dims)
    dkpe = rope_transpose(dkpe_r, saved["cos"], saved["sin"])
    return dict(dq=dq, dc=np.concatenate([dx, dkpe], axis=-1), dw=dW, dgamma=dgamma,
                dL=dLat, dkpe_r=dkpe_r)


# --------------------------------------------------------------------------
# Emulated sequence parallelism (Algorithm 1 steps 2, 3, 6; Section 5.2)
# --------------------------------------------------------------------------
def emulate_sp(P, q, c, w, gamma, cos, sin, dims: Dims, dO=None, form="laga"):
    """Run LAGA as P ranks inside one process and reassemble the result.

    Each rank r starts with the sequence chunk r of q and c (all heads).
    AllToAll_head(q) gives rank r the full sequence for heads
    H_r = [r n_h/P, (r+1) n_h/P); AllGather_seq(c) gives every rank the full
    latent; rank r runs ``forward``/``backward`` on its shard;
    AllToAll_seq(out) returns the sequence chunks with all heads.  In the
    backward the all-gather becomes a reduce-scatter (dc summed over ranks)
    and the head-sharded W_kv_b and gamma gradients are all-reduced (summed).
    ``dims`` describes the unsharded problem (dims.H = n_h).
    """
    n_h, S, B = dims.H, dims.S, dims.B
    assert n_h % P == 0 and S % P == 0
    Hr, Sr = n_h // P, S // P
    q = np.asarray(q, F64)
    c = np.asarray(c, F64)
    q_loc = [q[:, r * Sr:(r + 1) * Sr] for r in range(P)]      # seq-sharded input
    c_loc = [c[:, r * Sr:(r + 1) * Sr] for r in range(P)]
    c_gath = np.concatenate(c_loc, axis=1)                      # AllGather_seq
    fwd = forward if form == "laga" else forward_absorbed
    bwd = backward if form == "laga" else backward_absorbed
    outs, lses, grads = [], [], []
    for r in range(P):
        q_r = np.concatenate([ql[:, :, r * Hr:(r + 1) * Hr] for ql in q_loc], axis=1)
        d_r = dataclasses.replace(dims, H=Hr, head_offset=r * Hr, n_h_total=n_h)
        O_r, LSE_r, st = fwd(q_r, c_gath, w, gamma, cos, sin, d_r)
        outs.append(O_r)
        lses.append(LSE_r)
        if dO is not None:
            dO_r = np.asarray(dO, F64)[:, :, r * Hr:(r + 1) * Hr]
            grads.append(bwd(st, dO_r))
    # AllToAll_seq: rank r' keeps sequence chunk r' of every rank's heads.
    O_chunks = [np.concatenate([o[:, rp * Sr:(rp + 1) * Sr] for o in outs], axis=2)
                for rp in range(P)]
    res = dict(O=np.concatenate(O_chunks, axis=1), LSE=np.concatenate(lses, axis=1))
    if dO is None:
        return res
    res["dq"] = np.concatenate([g["dq"] for g in grads], axis=2)
    dc_full = sum(g["dc"] for g in grads)                       # reduce-scatter
    res["dc"] = np.concatenate([dc_full[:, rp * Sr:(rp + 1) * Sr] for rp in range(P)], axis=1)
    dh = dims.d_head_kv
    dw = np.zeros((dims.d_kv, n_h * dh))
    for r, g in enumerate(grads):                               # head-axis all-reduce
        dw[:, r * Hr * dh:(r + 1) * Hr * dh] += g["dw"]
    res["dw"] = dw
    res["dgamma"] = sum(g["dgamma"] for g in grads)
    return res


# --------------------------------------------------------------------------
# Closed forms: communication (Section 4.2, Table 1) and activation memory
# (Sections 1, 3.2, 3.3: n_h*d_kv absorbed intermediates versus per-head K/V)
# --------------------------------------------------------------------------
def comm_bytes_per_rank(form, S, P, n_h=128, d_nope=128, d_rope=64, d_v=128, d_kv=512):
    """Per-rank, per-forward sent bytes of each form.

    The page prints the values (Table 1) and the structural reason (B1's
    K-side all-to-all moves n_h(d_nope+d_v) elements per token, LAGA moves
    d_kv+d_rope) but no formula.  This reconstruction reproduces every cell
    of Table 1 and the n_h sweep of Section 4.2: each all-to-all sends the
    (P-1)/P off-rank part of (S/P) tokens x n_h x width at 4 bytes per
    element; explicit moves q (d_nope+d_rope), k (d_nope+d_rope), v (d_v) and
    out (d_v); LAGA and absorbed move q and out plus the latent gather
    counted as (d_kv+d_rope)/2 four-byte words per local token.
    """
    tok = S / P
    off = (P - 1) / P
    if form == "explicit":
        return 4.0 * tok * off * n_h * (2 * (d_nope + d_rope) + 2 * d_v)
    if form in ("laga", "absorbed"):
        return 4.0 * tok * (off * n_h * ((d_nope + d_rope) + d_v) + (d_kv + d_rope) / 2)
    raise ValueError(form)


def activation_elems_per_token(form, H, d_nope=128, d_v=128, d_kv=512):
    """Form-specific activation elements per token of one rank's shard.

    LAGA and explicit hold per-head K/V: H (d_nope + d_v).  Absorbed holds
    q_absorbed and the post-attention latent accumulator, each H d_kv.
    """
    if form in ("laga", "explicit"):
        return {"kv": H * (d_nope + d_v)}
    if form == "absorbed":
        return {"q_abs": H * d_kv, "o_lat": H * d_kv}
    raise ValueError(form)


def activation_bytes(form, S, H, elem_bytes=2, B=1, **kw):
    """Bytes of the form-specific activations for B*S tokens."""
    return B * S * elem_bytes * sum(activation_elems_per_token(form, H, **kw).values())
