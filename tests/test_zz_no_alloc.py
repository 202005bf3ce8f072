"""The allocation-free LayerNorm + RoPE backward entry point.

Callers that cannot allocate device memory (a runtime that has reserved the
whole device for its own pool, an embedding that owns only the tensors it
passes in) use laga_norm_rope_bwd_noalloc, which keeps its scratch in a
fixed array inside the library.  This test calls it through the C ABI on two
calls in a row of different sizes (the shared scratch keeps the previous
call's contents; the second uses the RMS variant of the latent norm) and
checks dc and dgamma against the fp64 oracle's norm backward and RoPE
transpose of the same upstream gradients, and
against what laga_bwd produced from them (only the recomputed LayerNorm
statistics differ, so the two agree to fp32 rounding).  The file name sorts
last so a run that stops at the first failure has already run every other
test.
"""

import numpy as np
import pytest
import torch

import oracle
from _harness import rel_fro, shard_of
from laga_inputs import as_f64, config, make_inputs

# fp32 arithmetic on exactly representable inputs: a few ulp per element,
# and the dgamma column sums over <= 1000 tokens
NOALLOC_REL_FRO = 1e-4

pytestmark = pytest.mark.gpu


def _ws(run, pass_, name, dtype, shape):
    ws = run.ws_saved if pass_ == 0 else run.ws_bwd
    for n, off, nb in run.workspace_tensors(pass_):
        if n == name:
            return ws[off:off + nb].view(dtype).view(*shape)
    raise KeyError(name)


def _oracle_norm_rope_bwd(cpu, wl, d_latent, d_kpe):
    """dc = [LayerNorm backward of d_latent | RoPE transpose of sum_h d_kpe]
    and dgamma, from the oracle in fp64."""
    c = as_f64(cpu["c"]).reshape(wl.B * wl.S, -1)
    d = oracle.Dims(S=wl.S, H=wl.H, norm=wl.norm)
    _, _, rstd, xhat = oracle.latent_norm(c[:, :wl.d_kv], as_f64(cpu["gamma"]), d)
    dx, dg = oracle.latent_norm_backward(as_f64(d_latent), xhat, rstd, as_f64(cpu["gamma"]), d)
    dk = as_f64(d_kpe).sum(axis=1).reshape(wl.B, wl.S, wl.d_rope)
    dkpe = oracle.rope_transpose(dk, as_f64(cpu["cos"]), as_f64(cpu["sin"]))
    dc = np.concatenate([dx.reshape(wl.B, wl.S, wl.d_kv), dkpe], axis=-1)
    return dc, dg


def test_noalloc_norm_rope_bwd_matches_oracle_on_two_calls():
    import sequence_latent_norm_gb300 as pkg
    lib = pkg._lib
    dev = torch.device("cuda:0")
    for wl in (config(1, S=1000, H=4), config(1, S=300, H=2, seed=77, B=2, norm="rms")):
        cpu = make_inputs(wl)
        t = {k: v.to(dev) for k, v in cpu.items()}
        run = pkg.Laga(shard_of(wl), device=dev)
        o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
        dq, dc_ref, dw, dg_ref = run.backward(t["q"], t["c"], t["w"], t["gamma"], t["cos"],
                                              t["sin"], o, lse, t["dO"])
        torch.cuda.synchronize()
        # the upstream gradients laga_bwd used: dL and each head's RoPE'd k_pe gradient
        T = wl.B * wl.S
        d_latent = _ws(run, 1, "dL", torch.float32, (T, 512)).clone()
        d_kpe = _ws(run, 1, "dk_pe_heads", torch.float32, (T, wl.H, 64)).clone()
        dc = torch.full_like(dc_ref, float("nan"))
        dg = torch.full_like(dg_ref, float("nan"))
        lib.norm_rope_bwd_noalloc(shard_of(wl).dims(), t["c"].data_ptr(), t["gamma"].data_ptr(),
                                  t["cos"].data_ptr(), t["sin"].data_ptr(), d_latent.data_ptr(),
                                  d_kpe.data_ptr(), dc.data_ptr(), dg.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
        lib.sync_check()
        dc_or, dg_or = _oracle_norm_rope_bwd(cpu, wl, d_latent.cpu(), d_kpe.cpu())
        for got, ref, orc, name in ((dc, dc_ref, dc_or, "dc"), (dg, dg_ref, dg_or, "dgamma")):
            g, r = as_f64(got), as_f64(ref)
            assert np.isfinite(g).all(), name
            e_or, e_self = rel_fro(g, orc), rel_fro(g, r)
            print(f"S={wl.S} B={wl.B} {wl.norm} {name}: rel-fro vs oracle {e_or:.2e}, "
                  f"vs laga_bwd {e_self:.2e}")
            assert e_or <= NOALLOC_REL_FRO, f"{name} rel-fro vs oracle {e_or:.3e}"
            assert e_self <= NOALLOC_REL_FRO, f"{name} rel-fro vs laga_bwd {e_self:.3e}"
