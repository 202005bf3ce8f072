"""The allocation-free LayerNorm + RoPE backward entry point.

Callers that cannot allocate device memory (a runtime that has reserved the
whole device for its own pool, an embedding that owns only the tensors it
passes in) use laga_norm_rope_bwd_noalloc, which keeps its scratch in a
fixed array inside the library.  This test calls it through the C ABI and
checks it against the dc and dgamma that laga_bwd produces from the same
upstream gradients, on two calls in a row of different sizes (the shared
scratch keeps the previous call's contents).  The file name sorts last so a
run that stops at the first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from _harness import GRAD_REL_FRO, rel_fro, shard_of
from laga_inputs import as_f64, config, make_inputs

pytestmark = pytest.mark.gpu


def _ws(run, pass_, name, dtype, shape):
    ws = run.ws_saved if pass_ == 0 else run.ws_bwd
    for n, off, nb in run.workspace_tensors(pass_):
        if n == name:
            return ws[off:off + nb].view(dtype).view(*shape)
    raise KeyError(name)


def test_noalloc_norm_rope_bwd_matches_laga_bwd_on_two_calls():
    import sequence_latent_norm_gb300 as pkg
    lib = pkg._lib
    dev = torch.device("cuda:0")
    for wl in (config(1, S=1000, H=4), config(1, S=300, H=2, seed=77)):
        t = {k: v.to(dev) for k, v in make_inputs(wl).items()}
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
        for got, ref, name in ((dc, dc_ref, "dc"), (dg, dg_ref, "dgamma")):
            g, r = as_f64(got), as_f64(ref)
            assert np.isfinite(g).all(), name
            assert rel_fro(g, r) <= GRAD_REL_FRO, f"{name} rel-fro {rel_fro(g, r):.3e}"
