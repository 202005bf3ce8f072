"""Shared helpers of the parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare."""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from laga_inputs import Workload, as_f64, make_inputs

# Tolerances for bf16 operands with fp32 accumulation.
O_MAX_ABS = 1e-2
O_REL_FRO = 5e-3
GRAD_REL_FRO = 1e-2
LSE_MAX_ABS = 2e-2


def rel_fro(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30))


def max_abs(x, y):
    return float(np.abs(np.asarray(x, np.float64) - np.asarray(y, np.float64)).max())


def shard_of(wl: Workload, form="laga", **over):
    import sequence_latent_norm_gb300 as pkg
    kw = dict(S=wl.S, H=wl.H, n_h_total=wl.n_h_total, head_offset=wl.head_offset, B=wl.B,
              d_nope=wl.d_nope, d_rope=wl.d_rope, d_v=wl.d_v, d_kv=wl.d_kv,
              io_dtype=wl.dtype, form=form)
    kw.update(over)
    return pkg.Shard(**kw)


def gpu_run(wl: Workload, cpu=None, form="laga", device="cuda:0", heads=None):
    """fwd + bwd of one shard on the GPU; returns CPU tensors.

    ``heads`` = (offset, count) runs a sub-shard of the workload's heads
    (the emulated SP rank), slicing q and dO accordingly.
    """
    import sequence_latent_norm_gb300 as pkg
    cpu = make_inputs(wl) if cpu is None else cpu
    dev = torch.device(device)
    t = {k: v.to(dev) for k, v in cpu.items()}
    if heads is not None:
        off, cnt = heads
        t["q"] = t["q"][:, :, off:off + cnt].contiguous()
        t["dO"] = t["dO"][:, :, off:off + cnt].contiguous()
        shard = shard_of(wl, form, H=cnt, head_offset=wl.head_offset + off)
    else:
        shard = shard_of(wl, form)
    run = pkg.Laga(shard, device=dev)
    o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
    dq, dc, dw, dg = run.backward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"], o, lse,
                                  t["dO"])
    pkg._lib.sync_check()
    return dict(O=o.cpu(), LSE=lse.cpu(), dq=dq.cpu(), dc=dc.cpu(), dw=dw.cpu(), dgamma=dg.cpu())


def oracle_dims(wl: Workload):
    return oracle.Dims(S=wl.S, H=wl.H, d_nope=wl.d_nope, d_rope=wl.d_rope, d_v=wl.d_v,
                       d_kv=wl.d_kv, B=wl.B, n_h_total=wl.n_h_total, head_offset=wl.head_offset)


def oracle_run(wl: Workload, cpu=None, heads=None):
    cpu = make_inputs(wl) if cpu is None else cpu
    a = {k: as_f64(v) for k, v in cpu.items()}
    d = oracle_dims(wl)
    O, LSE, st = oracle.forward(a["q"], a["c"], a["w"], a["gamma"], a["cos"], a["sin"], d,
                                heads=heads)
    g = oracle.backward(st, a["dO"])
    vmax = running_vmax(st["KV"][..., wl.d_nope:])
    # max over tokens j <= i and latent columns of |L_j|, broadcast to [B, S, 1, 1]
    lmax = np.maximum.accumulate(np.abs(st["L"]).max(axis=-1), axis=1)[:, :, None, None]
    return dict(O=O, LSE=LSE, dq=g["dq"], dc=g["dc"], dw=g["dw"], dgamma=g["dgamma"], vmax=vmax,
                lmax=lmax)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def o_abs_bound(Or, vmax):
    """Per-element max-abs bound on O: 1e-2, except where bf16 storage alone
    cannot resolve 1e-2.  O_i is a convex combination of the v_j (j <= i),
    which are stored in bf16 (half an ulp of |v_j|) and computed from the
    bf16-rounded normalised latent (about another half ulp); O is rounded
    to bf16 on output (half an ulp of |O|).  ``vmax`` is max_{j<=i} |v_jd|
    from the oracle, so the bound is max(1e-2, ulp(vmax) + ulp(|O|)/2)."""
    return np.maximum(O_MAX_ABS, bf16_ulp(vmax) + 0.5 * bf16_ulp(Or))


def running_vmax(v):
    """max over keys j <= i of |v[b, j, h, d]| (v: [B, S, H, d_v])."""
    return np.maximum.accumulate(np.abs(v), axis=1)


def check_forward(got, ref, where="", form="laga"):
    """O max-abs (per-element bound below), O relative Frobenius, LSE max-abs.

    The absorbed form stores one more intermediate in bf16: the latent
    accumulator o_lat_i, a convex combination of the L_j (j <= i), before
    the un-absorb product.  Its bound adds one bf16 ulp of the largest |L|
    the row averages (``lmax``)."""
    O, Or = as_f64(got["O"]), ref["O"]
    bound = o_abs_bound(Or, ref["vmax"])
    if form == "absorbed":
        bound = bound + bf16_ulp(ref["lmax"])
    excess = np.abs(O - Or) - bound
    assert excess.max() <= 0, (f"{where} O max-abs {max_abs(O, Or):.3e} exceeds its bound by "
                               f"{excess.max():.3e}")
    assert rel_fro(O, Or) <= O_REL_FRO, f"{where} O rel-fro {rel_fro(O, Or):.3e}"
    L, Lr = as_f64(got["LSE"]), ref["LSE"]
    assert max_abs(L, Lr) <= LSE_MAX_ABS, f"{where} LSE max-abs {max_abs(L, Lr):.3e}"


GRAD_ABS_RMS = 1e-4


def check_grads(got, ref, keys=("dq", "dc", "dw", "dgamma"), where=""):
    """Relative Frobenius error <= 1e-2, with an absolute floor of 1e-4 RMS
    per element for references that vanish (one token: dS = dO.v - dO.O = 0
    exactly, so dq is identically zero)."""
    for k in keys:
        g, r = as_f64(got[k]), ref[k]
        err = float(np.linalg.norm(g - r))
        lim = GRAD_REL_FRO * float(np.linalg.norm(r)) + GRAD_ABS_RMS * np.sqrt(r.size)
        assert err <= lim, f"{where} {k} rel-fro {rel_fro(g, r):.3e} (abs {err:.3e} > {lim:.3e})"


def head_slice(x, h, axis):
    return np.take(x, [h], axis=axis)


def dw_cols(wl: Workload, h):
    dh = wl.d_nope + wl.d_v
    return slice(h * dh, (h + 1) * dh)


def replace(wl: Workload, **kw):
    return dataclasses.replace(wl, **kw)
