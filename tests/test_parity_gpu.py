"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
identical seeded inputs, plus determinism and the explicit-form identity."""

import numpy as np
import pytest
import torch

from _harness import (check_forward, check_grads, dw_cols, gpu_run, head_view, oracle_run,
                      shard_of)
from laga_inputs import as_f64, config, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    dict(S=200, H=2),                 # ragged: several 64/128 tiles plus a tail
    dict(S=1, H=1),                   # a single token
    dict(S=129, H=3, B=2),            # batch > 1, one past a tile edge
    dict(S=384, H=2, n_h_total=5, head_offset=3),  # shard inside a wider W_kv_b
])
def test_small_canonical_dims_match_oracle(case):
    wl = config(1, **case)
    got = gpu_run(wl)
    ref = oracle_run(wl)
    check_forward(got, ref, str(case))
    check_grads(got, ref, where=str(case))


@pytest.mark.parametrize("case", [
    dict(S=200, H=2, d_nope=64, d_rope=32, d_v=64, d_kv=256),   # all dims below canonical
    dict(S=150, H=3, d_kv=256),                                  # canonical heads, narrower latent
])
def test_noncanonical_bf16_dims_match_oracle(case):
    """bf16 I/O with dims other than 128/64/128/512: zero-padded into the
    canonical layout on device, with dq converted by dq_final."""
    wl = config(1, **case)
    got = gpu_run(wl)
    ref = oracle_run(wl)
    check_forward(got, ref, str(case))
    check_grads(got, ref, where=str(case))


def test_tiny_fp32_config_sp1_and_sp2():
    wl = config(0)
    cpu = make_inputs(wl)
    ref = oracle_run(wl, cpu)
    got = gpu_run(wl, cpu)
    check_forward(got, ref, "sp1")
    check_grads(got, ref, where="sp1")
    # emulated SP=2: rank r runs heads [2r, 2r+2) over the full sequence; O,
    # LSE, dq and dW are concatenated over heads, dc and dgamma summed.
    parts = [gpu_run(wl, cpu, heads=(2 * r, 2)) for r in range(2)]
    sp = dict(O=torch.cat([p["O"] for p in parts], 2), LSE=torch.cat([p["LSE"] for p in parts], 1),
              dq=torch.cat([p["dq"] for p in parts], 2), dw=torch.cat([p["dw"] for p in parts], 1),
              dc=parts[0]["dc"] + parts[1]["dc"], dgamma=parts[0]["dgamma"] + parts[1]["dgamma"])
    check_forward(sp, ref, "sp2")
    check_grads(sp, ref, where="sp2")
    # head-local results do not depend on the sharding
    assert torch.equal(sp["O"], got["O"]) and torch.equal(sp["dq"], got["dq"])


def test_config1_full_compare():
    wl = config(1)
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu)
    ref = oracle_run(wl, cpu)
    check_forward(got, ref, "config1")
    check_grads(got, ref, where="config1")


def test_config2_full_size_all_heads():
    """S=16384, the 16-head shard the bench times, in the same launch
    configuration: every output of every head -- O, LSE, dq, dc, dW and
    dgamma -- element by element against the oracle's full fwd + bwd."""
    wl = config(2)
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu)
    ref = oracle_run(wl, cpu)
    check_forward(got, ref, "config2 S=16384")
    check_grads(got, ref, where="config2 S=16384")


def test_sweep_largest_point_sampled_heads():
    """The largest point of the S x H sweep (S=32768, 32-head shard): the
    widest grid (256 query tiles x 32 heads) and the largest workspace
    offsets, against the oracle on the first and last heads (O, LSE, dq and
    their columns of dW_kv_b)."""
    wl = config(4, S=32768, H=32, n_h_total=32)
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu)
    hs = [0, 31]
    ref = oracle_run(wl, cpu, heads=hs)
    for h in hs:
        g, r = head_view(got, ref, h)
        check_forward(g, r, f"S=32768 H=32 head {h}")
        cols = dw_cols(wl, h)
        check_grads(dict(dq=got["dq"][:, :, h], dw=got["dw"][:, cols]),
                    dict(dq=ref["dq"][:, :, h], dw=ref["dw"][:, cols]), keys=("dq", "dw"),
                    where=f"S=32768 H=32 head {h}")


def test_emulated_sp8_matches_oracle_on_config1_dims():
    """Emulated SP = 8 over a 16-head layer (2 heads per rank, full S): head-
    local outputs concatenate, dc and dgamma partials sum (Section 5.2)."""
    wl = config(1, S=1024)
    cpu = make_inputs(wl)
    ref = oracle_run(wl, cpu)
    parts = [gpu_run(wl, cpu, heads=(2 * r, 2)) for r in range(8)]
    sp = dict(O=torch.cat([p["O"] for p in parts], 2), LSE=torch.cat([p["LSE"] for p in parts], 1),
              dq=torch.cat([p["dq"] for p in parts], 2), dw=torch.cat([p["dw"] for p in parts], 1),
              dc=sum(p["dc"] for p in parts), dgamma=sum(p["dgamma"] for p in parts))
    check_forward(sp, ref, "sp8")
    check_grads(sp, ref, where="sp8")


def test_run_to_run_bitwise_determinism():
    wl = config(1, S=1000, H=4)
    cpu = make_inputs(wl)
    a, b = gpu_run(wl, cpu), gpu_run(wl, cpu)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_laga_equals_explicit_form_bitwise_at_sp1():
    """Proposition 1 / Section 4.5: same matmuls, reordered K/V views.
    Full-head SP=1 run (S=4096, n_h=128); both forms also against the oracle
    on sampled heads."""
    wl = config(3)
    cpu = make_inputs(wl)
    a = gpu_run(wl, cpu, form="laga")
    b = gpu_run(wl, cpu, form="explicit")
    for k in a:
        assert torch.equal(a[k], b[k]), k
    hs = [0, 77]
    ref = oracle_run(wl, cpu, heads=hs)
    for h in hs:
        g, r = head_view(a, ref, h)
        check_forward(g, r, f"config3 head {h}")
        cols = dw_cols(wl, h)
        check_grads(dict(dq=a["dq"][:, :, h], dw=a["dw"][:, cols]),
                    dict(dq=ref["dq"][:, :, h], dw=ref["dw"][:, cols]), keys=("dq", "dw"),
                    where=f"config3 head {h}")


def test_laga_equals_explicit_form_bitwise_on_ragged_batch():
    """The identity of the two forms on a ragged length, B = 2 and a shard
    inside a wider W_kv_b, and both against the oracle."""
    wl = config(1, S=333, H=3, B=2, n_h_total=7, head_offset=2)
    cpu = make_inputs(wl)
    a = gpu_run(wl, cpu, form="laga")
    b = gpu_run(wl, cpu, form="explicit")
    for k in a:
        assert torch.equal(a[k], b[k]), k
    ref = oracle_run(wl, cpu)
    check_forward(a, ref, "ragged laga")
    check_grads(a, ref, where="ragged laga")


@pytest.mark.parametrize("form", ["laga", "laga_fused"])
def test_bwd_overlap_entry_point_is_bitwise_equal_to_laga_bwd(form):
    """laga_bwd_overlap (the dQ kernel on a second stream of the caller's)
    computes exactly what laga_bwd does on one stream, and orders its work
    before what follows on the compute stream.  The fused form's dQ kernel
    reads the K/V its dK/dV kernel rebuilds, so there the call keeps stream
    order; the results are the same."""
    import sequence_latent_norm_gb300 as pkg
    wl = config(1, S=1000, H=4)
    dev = torch.device("cuda:0")
    t = {k: v.to(dev) for k, v in make_inputs(wl).items()}
    run = pkg.Laga(shard_of(wl, form), device=dev)
    o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
    a = run.backward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"], o, lse, t["dO"])
    a = [x.clone() for x in a]
    aux = torch.cuda.Stream(dev)
    for _ in range(2):
        b = run.backward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"], o, lse, t["dO"],
                         aux_stream=aux)
        b = [x.clone() for x in b]      # on the compute stream: after the join
        pkg._lib.sync_check()
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("wl,form", [
    (config(1, S=333, H=3, B=2, n_h_total=7, head_offset=2, norm="rms"), "laga"),
    (config(1, S=1000, H=4, norm="rms"), "laga"),
    (config(1, S=200, H=2, norm="rms"), "absorbed"),
    (config(0, norm="rms"), "laga"),
    (config(1, S=150, H=3, d_kv=256, norm="rms"), "laga"),
], ids=["ragged-B2", "S1000", "absorbed", "tiny-fp32", "dkv256"])
def test_rms_latent_norm_variant_matches_oracle(wl, form):
    """The RMS variant of the latent norm (no centring) through the whole
    path: forward, dq, dc, dW and dgamma against the oracle's rmsnorm."""
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu, form=form)
    ref = oracle_run(wl, cpu)
    check_forward(got, ref, f"rms {wl.name} S={wl.S}", form=form)
    check_grads(got, ref, where=f"rms {wl.name} S={wl.S}")


FUSED_CASES = [
    dict(S=200, H=2),                                # ragged tail
    dict(S=1, H=1),                                  # a single token
    dict(S=129, H=3, B=2),                           # batch > 1, one past a tile edge
    dict(S=384, H=2, n_h_total=5, head_offset=3),    # shard inside a wider W_kv_b
    dict(S=150, H=3, d_kv=256),                      # narrower latent (padded W and L)
    dict(S=333, H=2, norm="rms"),                    # RMS latent norm
    dict(S=4096, H=16),                              # the 4096-token, 16-head shard
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_fused_upprojection_form_matches_oracle_and_equals_laga(case):
    """The fused form rebuilds each key tile's k_nope | v = L_j W_h inside
    the key-stationary backward instead of reading the forward's K/V.  The
    rebuild accumulates the same 32 K-steps in the same order as the
    up-projection GEMM and rounds to bf16 the same way, so every output is
    bit-identical to the LAGA form; both are checked against the oracle."""
    wl = config(1, **case)
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu, form="laga_fused")
    ref = oracle_run(wl, cpu)
    check_forward(got, ref, f"fused {case}")
    check_grads(got, ref, where=f"fused {case}")
    base = gpu_run(wl, cpu, form="laga")
    for k in got:
        assert torch.equal(got[k], base[k]), f"fused form differs from LAGA in {k}"


def test_fused_form_fp32_config_equals_laga():
    wl = config(0)
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu, form="laga_fused")
    check_forward(got, oracle_run(wl, cpu), "fused fp32-config0")
    base = gpu_run(wl, cpu, form="laga")
    for k in got:
        assert torch.equal(got[k], base[k]), k


@pytest.mark.parametrize("S,H", [(16384, 16), (32768, 32)])
def test_fused_form_full_size_equals_laga(S, H):
    """At the full shard (S=16384, 16 heads, the benchmarked launch) and at
    the sweep's largest point (S=32768, 32 heads), where the LAGA form
    itself is checked against the oracle: the fused form's outputs are
    bit-identical to it."""
    wl = config(2) if S == 16384 else config(4, S=S, H=H, n_h_total=H)
    cpu = make_inputs(wl)
    got = gpu_run(wl, cpu, form="laga_fused")
    base = gpu_run(wl, cpu, form="laga")
    for k in got:
        assert torch.equal(got[k], base[k]), f"fused form differs from LAGA in {k} at S={S}"
