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
    return dict(O=O, LSE=LSE, dq=g["dq"], dc=g["dc"], dw=g["dw"], dgamma=g["dgamma"])


def check_forward(got, ref, where=""):
    O, Or = as_f64(got["O"]), ref["O"]
    assert max_abs(O, Or) <= O_MAX_ABS, f"{where} O max-abs {max_abs(O, Or):.3e}"
    assert rel_fro(O, Or) <= O_REL_FRO, f"{where} O rel-fro {rel_fro(O, Or):.3e}"
    L, Lr = as_f64(got["LSE"]), ref["LSE"]
    assert max_abs(L, Lr) <= LSE_MAX_ABS, f"{where} LSE max-abs {max_abs(L, Lr):.3e}"


def check_grads(got, ref, keys=("dq", "dc", "dw", "dgamma"), where=""):
    for k in keys:
        e = rel_fro(as_f64(got[k]), ref[k])
        assert e <= GRAD_REL_FRO, f"{where} {k} rel-fro {e:.3e}"


def head_slice(x, h, axis):
    return np.take(x, [h], axis=axis)


def dw_cols(wl: Workload, h):
    dh = wl.d_nope + wl.d_v
    return slice(h * dh, (h + 1) * dh)


def replace(wl: Workload, **kw):
    return dataclasses.replace(wl, **kw)
