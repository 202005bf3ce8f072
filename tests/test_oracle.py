"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against brute force on tiny inputs, a library
routine the method reduces to, a closed form, an invariant, or a value the
LAGA paper page prints.  None of these re-types the oracle's own formula.
"""

import dataclasses
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc
from oracle.laga import Dims

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(rng, dims: Dims, scale_q=1.0):
    q = rng.standard_normal((dims.B, dims.S, dims.H, dims.d_qk)) * scale_q
    c = rng.standard_normal((dims.B, dims.S, dims.d_kv + dims.d_rope))
    w = rng.standard_normal((dims.d_kv, dims.n_total * dims.d_head_kv)) / math.sqrt(dims.d_kv)
    gamma = 1.0 + 0.1 * rng.standard_normal(dims.d_kv)
    cos, sin = orc.rope_tables(dims.S, dims.d_rope)
    dO = rng.standard_normal((dims.B, dims.S, dims.H, dims.d_v))
    return q, c, w, gamma, cos, sin, dO


TINY = Dims(S=5, H=2, d_nope=4, d_rope=4, d_v=3, d_kv=6, B=2, n_h_total=3, head_offset=1)


# ----------------------------------------------------------------- brute force
def _brute_forward(q, c, w, gamma, dims: Dims, theta=10000.0):
    """Scalar Python loops over the definitions, with its own RoPE angles."""
    B, S, H = dims.B, dims.S, dims.H
    dn, dr, dv, dk = dims.d_nope, dims.d_rope, dims.d_v, dims.d_kv
    dh = dn + dv
    half = dr // 2
    O = np.zeros((B, S, H, dv))
    LSE = np.zeros((B, H, S))

    def rot(vec, t):
        out = [0.0] * dr
        for i in range(half):
            a = t * theta ** (-2.0 * i / dr)
            out[i] = vec[i] * math.cos(a) - vec[i + half] * math.sin(a)
            out[i + half] = vec[i + half] * math.cos(a) + vec[i] * math.sin(a)
        return out

    for b in range(B):
        Lrows, kpe = [], []
        for t in range(S):
            x = [c[b, t, k] for k in range(dk)]
            mu = sum(x) / dk
            var = sum((xi - mu) ** 2 for xi in x) / dk
            Lrows.append([(x[k] - mu) / math.sqrt(var + dims.eps) * gamma[k] for k in range(dk)])
            kpe.append(rot([c[b, t, dk + i] for i in range(dr)], t))
        for h in range(H):
            col0 = (dims.head_offset + h) * dh
            kn = [[sum(Lrows[t][k] * w[k, col0 + d] for k in range(dk)) for d in range(dn)]
                  for t in range(S)]
            vv = [[sum(Lrows[t][k] * w[k, col0 + dn + d] for k in range(dk)) for d in range(dv)]
                  for t in range(S)]
            for i in range(S):
                qn = [q[b, i, h, d] for d in range(dn)]
                qr = rot([q[b, i, h, dn + d] for d in range(dr)], i)
                s = []
                for j in range(i + 1):
                    dot = sum(qn[d] * kn[j][d] for d in range(dn)) + \
                        sum(qr[d] * kpe[j][d] for d in range(dr))
                    s.append(dot / math.sqrt(dn + dr))
                m = max(s)
                e = [math.exp(x - m) for x in s]
                tot = sum(e)
                LSE[b, h, i] = m + math.log(tot)
                for d in range(dv):
                    O[b, i, h, d] = sum(e[j] / tot * vv[j][d] for j in range(i + 1))
    return O, LSE


def test_forward_matches_brute_force_loops():
    rng = np.random.default_rng(0)
    q, c, w, gamma, cos, sin, _ = _rand_problem(rng, TINY)
    O, LSE, _ = orc.forward(q, c, w, gamma, cos, sin, TINY)
    O_b, LSE_b = _brute_forward(q, c, w, gamma, TINY)
    np.testing.assert_allclose(O, O_b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, LSE_b, rtol=0, atol=1e-12)


def test_forward_block_size_does_not_matter():
    rng = np.random.default_rng(1)
    d = Dims(S=37, H=2, d_nope=8, d_rope=4, d_v=8, d_kv=16)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, d)
    O1, L1, s1 = orc.forward(q, c, w, gamma, cos, sin, d, block=512)
    O2, L2, s2 = orc.forward(q, c, w, gamma, cos, sin, d, block=5)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)
    g1, g2 = orc.backward(s1, dO), orc.backward(s2, dO, block=7)
    for k in ("dq", "dc", "dw", "dgamma"):
        np.testing.assert_allclose(g1[k], g2[k], atol=1e-12)


# ----------------------------------------------------------------- RoPE
def test_rope_tables_against_math_and_identity_at_position_zero():
    cos, sin = orc.rope_tables(9, 6, theta=10000.0)
    for t in range(9):
        for i in range(3):
            a = t * 10000.0 ** (-2.0 * i / 6)
            assert cos[t, i] == pytest.approx(math.cos(a), abs=1e-15)
            assert sin[t, i] == pytest.approx(math.sin(a), abs=1e-15)
    x = np.random.default_rng(2).standard_normal((1, 9, 6))
    y = orc.rope(x, cos, sin)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])             # position 0: identity
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1),
                               rtol=1e-14)                       # rotation keeps norms
    np.testing.assert_allclose(orc.rope_transpose(y, cos, sin), x, atol=1e-14)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(3)
    d = Dims(S=12, H=1, d_nope=4, d_rope=8, d_v=4, d_kv=8)
    q, c, w, gamma, _, _, _ = _rand_problem(rng, d)
    c0, s0 = orc.rope_tables(d.S, d.d_rope, pos0=0)
    c7, s7 = orc.rope_tables(d.S, d.d_rope, pos0=7)
    O0, L0, _ = orc.forward(q, c, w, gamma, c0, s0, d)
    O7, L7, _ = orc.forward(q, c, w, gamma, c7, s7, d)
    np.testing.assert_allclose(O0, O7, atol=1e-12)
    np.testing.assert_allclose(L0, L7, atol=1e-12)


# ----------------------------------------------------------------- LayerNorm
def test_layernorm_matches_torch_and_is_affine_invariant():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 7, 16))
    g = 1.0 + 0.1 * rng.standard_normal(16)
    L, mean, rstd, xhat = orc.layernorm(x, g, 1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (16,), weight=torch.from_numpy(g),
                                         bias=None, eps=1e-5).numpy()
    np.testing.assert_allclose(L, ref, atol=1e-13)
    L2, _, _, _ = orc.layernorm(3.5 * x - 2.0, g, 0.0)
    L3, _, _, _ = orc.layernorm(x, g, 0.0)
    np.testing.assert_allclose(L2, L3, atol=1e-12)


def test_rmsnorm_matches_torch_and_is_scale_but_not_shift_invariant():
    """The RMS variant of the latent norm: torch's rms_norm; invariant to a
    positive scale of x (eps = 0), but, having no centring, not to a shift
    (a LayerNorm by mistake would be)."""
    rng = np.random.default_rng(40)
    x = rng.standard_normal((3, 7, 16))
    g = 1.0 + 0.1 * rng.standard_normal(16)
    L, mean, rstd, xhat = orc.rmsnorm(x, g, 1e-5)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (16,), weight=torch.from_numpy(g),
                                       eps=1e-5).numpy()
    np.testing.assert_allclose(L, ref, atol=1e-13)
    assert np.all(mean == 0.0)
    L2, _, _, _ = orc.rmsnorm(3.5 * x, g, 0.0)
    L3, _, _, _ = orc.rmsnorm(x, g, 0.0)
    np.testing.assert_allclose(L2, L3, atol=1e-12)
    L4, _, _, _ = orc.rmsnorm(x + 2.0, g, 0.0)
    assert np.abs(L4 - L3).max() > 0.1


# ----------------------------------------------------------------- closed forms
def test_zero_query_gives_running_mean_and_log_count():
    rng = np.random.default_rng(5)
    d = Dims(S=9, H=2, d_nope=4, d_rope=4, d_v=5, d_kv=8)
    _, c, w, gamma, cos, sin, _ = _rand_problem(rng, d)
    q = np.zeros((1, d.S, d.H, d.d_qk))
    O, LSE, st = orc.forward(q, c, w, gamma, cos, sin, d)
    v = st["KV"][..., d.d_nope:]
    for i in range(d.S):
        np.testing.assert_allclose(O[0, i], v[0, :i + 1].mean(axis=0), atol=1e-13)
        np.testing.assert_allclose(LSE[0, :, i], math.log(i + 1), atol=1e-13)


def test_first_row_sees_only_itself():
    rng = np.random.default_rng(6)
    d = Dims(S=6, H=3, d_nope=4, d_rope=4, d_v=5, d_kv=8)
    q, c, w, gamma, cos, sin, _ = _rand_problem(rng, d)
    O, LSE, st = orc.forward(q, c, w, gamma, cos, sin, d)
    v = st["KV"][0, 0, :, d.d_nope:]
    kn = st["KV"][0, 0, :, :d.d_nope]
    np.testing.assert_allclose(O[0, 0], v, atol=1e-14)
    # position 0: RoPE is the identity, so s_00 uses the raw rope bands
    s00 = (np.einsum("hd,hd->h", q[0, 0, :, :d.d_nope], kn)
           + q[0, 0, :, d.d_nope:] @ c[0, 0, d.d_kv:]) / math.sqrt(d.d_qk)
    np.testing.assert_allclose(LSE[0, :, 0], s00, atol=1e-13)


def test_lse_normalises_every_row():
    rng = np.random.default_rng(7)
    d = Dims(S=20, H=2, d_nope=8, d_rope=4, d_v=8, d_kv=8)
    q, c, w, gamma, cos, sin, _ = _rand_problem(rng, d, scale_q=3.0)
    _, LSE, st = orc.forward(q, c, w, gamma, cos, sin, d)
    kn = st["KV"][..., :d.d_nope]
    for h in range(d.H):
        s = (st["q_nope"][0, :, h] @ kn[0, :, h].T + st["q_rope_r"][0, :, h] @ st["kpe_r"][0].T)
        s = s / math.sqrt(d.d_qk)
        s[np.triu_indices(d.S, 1)] = -np.inf
        np.testing.assert_allclose(np.exp(s - LSE[0, h][:, None]).sum(axis=1), 1.0, atol=1e-13)


# ----------------------------------------------------------------- library reduction
@pytest.mark.parametrize("norm", ["layer", "rms"])
def test_no_rope_case_reduces_to_torch_sdpa_forward_and_autograd(norm):
    """d_rope = 0: the method is causal SDPA over (q, N(x) W^k, N(x) W^v),
    N = LayerNorm or its RMS variant."""
    rng = np.random.default_rng(8)
    d = Dims(S=11, H=2, d_nope=8, d_rope=0, d_v=6, d_kv=10, norm=norm)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, d)
    O, LSE, st = orc.forward(q, c, w, gamma, cos, sin, d)
    g = orc.backward(st, dO)

    tq = torch.tensor(q, requires_grad=True)
    tc = torch.tensor(c, requires_grad=True)
    tw = torch.tensor(w, requires_grad=True)
    tg = torch.tensor(gamma, requires_grad=True)
    if norm == "rms":
        L = torch.nn.functional.rms_norm(tc, (d.d_kv,), weight=tg, eps=d.eps)
    else:
        L = torch.nn.functional.layer_norm(tc, (d.d_kv,), weight=tg, bias=None, eps=d.eps)
    kv = (L @ tw).view(1, d.S, d.H, d.d_head_kv)
    k, v = kv[..., :d.d_nope], kv[..., d.d_nope:]
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), is_causal=True)
    o = o.transpose(1, 2)
    (o * torch.tensor(dO)).sum().backward()
    np.testing.assert_allclose(O, o.detach().numpy(), atol=1e-12)
    s = torch.einsum("bihd,bjhd->bhij", tq, k) / math.sqrt(d.d_qk)
    s = s.masked_fill(torch.ones(d.S, d.S, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(LSE, torch.logsumexp(s, dim=-1).detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(g["dq"], tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dc"], tc.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dw"], tw.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dgamma"], tg.grad.numpy(), atol=1e-11)


# ----------------------------------------------------------------- finite differences
FD = Dims(S=6, H=2, d_nope=4, d_rope=4, d_v=3, d_kv=6, B=1, n_h_total=3, head_offset=1)


def _loss(q, c, w, gamma, cos, sin, dO, dims):
    O, _, _ = orc.forward(q, c, w, gamma, cos, sin, dims)
    return float((O * dO).sum())


@pytest.mark.parametrize("norm", ["layer", "rms"])
@pytest.mark.parametrize("name", ["q", "c", "w", "gamma"])
def test_backward_matches_central_differences(name, norm):
    rng = np.random.default_rng(9)
    FD_ = dataclasses.replace(FD, norm=norm)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, FD_)
    args = dict(q=q, c=c, w=w, gamma=gamma)
    _, _, st = orc.forward(q, c, w, gamma, cos, sin, FD_)
    g = orc.backward(st, dO)
    analytic = {"q": g["dq"], "c": g["dc"], "gamma": g["dgamma"]}
    if name == "w":
        full = np.zeros_like(w)
        dh = FD.d_head_kv
        full[:, FD.head_offset * dh:(FD.head_offset + FD.H) * dh] = g["dw"]
        analytic["w"] = full
    x = args[name]
    num = np.zeros_like(x)
    h = 1e-6
    for idx in np.ndindex(x.shape):
        old = x[idx]
        x[idx] = old + h
        fp = _loss(dO=dO, cos=cos, sin=sin, dims=FD_, **args)
        x[idx] = old - h
        fm = _loss(dO=dO, cos=cos, sin=sin, dims=FD_, **args)
        x[idx] = old
        num[idx] = (fp - fm) / (2 * h)
    err = np.linalg.norm(analytic[name] - num) / max(np.linalg.norm(num), 1e-30)
    assert err < 1e-7, err


# ----------------------------------------------------------------- invariants
def test_constant_latent_makes_output_independent_of_queries():
    """Equal latents give equal v_j, so O_i = v whatever the scores are:
    dq must vanish, which needs dS_ij = P_ij (dP_ij - delta_i) to cancel
    exactly (sum_j dS_ij = 0 with dP_ij = delta_i)."""
    rng = np.random.default_rng(10)
    d = Dims(S=10, H=2, d_nope=6, d_rope=4, d_v=5, d_kv=8)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, d)
    c[:, :, :d.d_kv] = c[:, :1, :d.d_kv]          # every token has the same latent
    O, _, st = orc.forward(q, c, w, gamma, cos, sin, d)
    np.testing.assert_allclose(O, np.broadcast_to(O[:, :1], O.shape), atol=1e-14)
    g = orc.backward(st, dO)
    assert np.abs(g["dq"]).max() < 1e-13
    assert np.abs(g["dc"][..., d.d_kv:]).max() < 1e-13   # k_pe only reaches O via P
    assert np.abs(g["dw"]).max() > 1e-2                  # v still carries gradient


def test_latent_gradient_sums_to_zero_over_features():
    rng = np.random.default_rng(11)
    d = Dims(S=14, H=3, d_nope=8, d_rope=4, d_v=8, d_kv=12)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, d)
    _, _, st = orc.forward(q, c, w, gamma, cos, sin, d)
    g = orc.backward(st, dO)
    assert np.abs(g["dc"][..., :d.d_kv].sum(axis=-1)).max() < 1e-12


# ----------------------------------------------------------------- Propositions 1-2
def test_absorbed_form_equals_explicit_form():
    rng = np.random.default_rng(12)
    d = Dims(S=19, H=3, d_nope=8, d_rope=4, d_v=6, d_kv=16, n_h_total=4, head_offset=1)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, d)
    O, LSE, st = orc.forward(q, c, w, gamma, cos, sin, d)
    Oa, LSEa, sta = orc.forward_absorbed(q, c, w, gamma, cos, sin, d)
    np.testing.assert_allclose(Oa, O, atol=1e-12)
    np.testing.assert_allclose(LSEa, LSE, atol=1e-12)
    g, ga = orc.backward(st, dO), orc.backward_absorbed(sta, dO)
    for k in ("dq", "dc", "dw", "dgamma"):
        np.testing.assert_allclose(ga[k], g[k], atol=1e-11, err_msg=k)


@pytest.mark.parametrize("P", [2, 4])
@pytest.mark.parametrize("form", ["laga", "absorbed"])
def test_emulated_sp_equals_unsharded(P, form):
    rng = np.random.default_rng(13)
    d = Dims(S=16, H=8, d_nope=8, d_rope=4, d_v=8, d_kv=16)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, d)
    O, LSE, st = orc.forward(q, c, w, gamma, cos, sin, d)
    g = orc.backward(st, dO)
    r = orc.emulate_sp(P, q, c, w, gamma, cos, sin, d, dO=dO, form=form)
    np.testing.assert_allclose(r["O"], O, atol=1e-12)
    np.testing.assert_allclose(r["LSE"], LSE, atol=1e-12)
    for k in ("dq", "dc", "dw", "dgamma"):
        np.testing.assert_allclose(r[k], g[k], atol=1e-11, err_msg=k)


def test_head_subset_matches_full_shard():
    rng = np.random.default_rng(14)
    d = Dims(S=12, H=4, d_nope=8, d_rope=4, d_v=8, d_kv=16)
    q, c, w, gamma, cos, sin, dO = _rand_problem(rng, d)
    O, LSE, st = orc.forward(q, c, w, gamma, cos, sin, d)
    g = orc.backward(st, dO)
    Os, LSEs, sts = orc.forward(q, c, w, gamma, cos, sin, d, heads=[2])
    gs = orc.backward(sts, dO)
    np.testing.assert_array_equal(Os[:, :, 2], O[:, :, 2])
    np.testing.assert_array_equal(LSEs[:, 2], LSE[:, 2])
    np.testing.assert_allclose(gs["dq"][:, :, 2], g["dq"][:, :, 2], atol=1e-14)
    cols = slice(2 * d.d_head_kv, 3 * d.d_head_kv)
    np.testing.assert_allclose(gs["dw"][:, cols], g["dw"][:, cols], atol=1e-13)
    assert np.isnan(Os[:, :, 0]).all() and gs["dc"] is None


# ----------------------------------------------------------------- printed values
def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


def test_comm_closed_form_reproduces_table1():
    rows = _read_table("table1_comm_mb.txt")
    assert len(rows) == 8
    for sp, S, b1, b2, laga in rows:
        assert round(orc.comm_bytes_per_rank("explicit", S, int(sp)) / 1e6, 1) == b1
        assert round(orc.comm_bytes_per_rank("absorbed", S, int(sp)) / 1e6, 1) == b2
        assert round(orc.comm_bytes_per_rank("laga", S, int(sp)) / 1e6, 1) == laga


def test_comm_ratio_versus_heads_matches_section_4_2():
    for n_h, ratio in _read_table("comm_ratio_vs_heads.txt"):
        r = (orc.comm_bytes_per_rank("explicit", 8192, 8, n_h=int(n_h))
             / orc.comm_bytes_per_rank("laga", 8192, 8, n_h=int(n_h)))
        assert round(r, 2) == ratio


def test_activation_closed_form_ratio():
    # per tensor the absorbed intermediate is d_kv / (d_nope + d_v) = 2x the
    # per-head K/V at DeepSeek-V3 dims; it is larger whenever d_kv > d_head.
    la = orc.activation_elems_per_token("laga", 16)
    ab = orc.activation_elems_per_token("absorbed", 16)
    assert ab["q_abs"] == ab["o_lat"] == 2 * la["kv"] == 16 * 512
    assert orc.activation_bytes("absorbed", 16384, 16) - orc.activation_bytes("laga", 16384, 16) \
        == 16384 * 2 * (2 * 16 * 512 - 16 * 256)


# ----------------------------------------------------------------- shared inputs
def test_seeded_inputs_have_the_stated_distributions():
    from laga_inputs import config, make_inputs, as_f64
    wl = config(1, S=512)
    a, b = make_inputs(wl), make_inputs(wl)
    for k in a:
        assert torch.equal(a[k], b[k])
    w = as_f64(a["w"])
    assert abs(w.std() - 1 / math.sqrt(512)) < 0.01 / math.sqrt(512) * 10
    assert abs(as_f64(a["gamma"]).std() - 0.1) < 0.02
    cos, sin = orc.rope_tables(wl.S, wl.d_rope)
    np.testing.assert_allclose(as_f64(a["cos"]), cos, atol=1e-7)
    np.testing.assert_allclose(as_f64(a["sin"]), sin, atol=1e-7)
    assert a["q"].dtype == torch.bfloat16 and config(0).dtype == "fp32"
