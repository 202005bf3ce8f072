"""The absorbed-form contrast path (Section 3.2, B2) on the GPU: same
function as LAGA (Propositions 1-2), different activation memory."""

import numpy as np
import pytest
import torch

import oracle
from _harness import check_forward, check_grads, gpu_run, oracle_run, shard_of
from laga_inputs import config, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [config(1, S=200, H=2), config(0)], ids=["v3-ragged", "tiny-fp32"])
def test_absorbed_form_matches_oracle(wl):
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu, form="absorbed")
    ref = oracle_run(wl, cpu)
    check_forward(got, ref, "absorbed", form="absorbed")
    check_grads(got, ref, where="absorbed")


def _peak_after_forward(wl, form, cpu):
    import sequence_latent_norm_gb300 as pkg
    dev = torch.device("cuda:0")
    t = {k: v.to(dev) for k, v in cpu.items()}
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    run = pkg.Laga(shard_of(wl, form), device=dev)
    o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
    torch.cuda.synchronize()
    pkg._lib.sync_check()
    peak = torch.cuda.max_memory_allocated(dev) - base
    del run, o, lse
    return peak


@pytest.mark.parametrize("S,H", [(2048, 8), (4096, 16), (8192, 16), (32768, 32)])
def test_measured_activation_gap_matches_closed_form(S, H):
    """Peak device memory of a forward (saved activations + outputs): the
    absorbed form exceeds LAGA by exactly its n_h*d_kv intermediates minus
    the per-head K/V they replace, within allocator granularity."""
    wl = config(1, S=S, H=H, n_h_total=H)
    cpu = make_inputs(wl, with_grad_out=False)
    gap = _peak_after_forward(wl, "absorbed", cpu) - _peak_after_forward(wl, "laga", cpu)
    closed = oracle.activation_bytes("absorbed", S, H) - oracle.activation_bytes("laga", S, H)
    assert abs(gap - closed) <= max(2 << 20, 0.01 * closed), (gap, closed)
