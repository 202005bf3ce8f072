"""Pins of the attention-block oracle (oracle/block.py) to things other than
itself: central finite differences of its forward for every input and
weight, and, with selection matrices as the projections, the per-rank
oracle's own forward and backward (so the reshapes, the head order and the
transposes of the three projections are fixed)."""

import dataclasses
import math

import numpy as np
import pytest

import oracle
from oracle.block import block_backward, block_forward

TINY = oracle.Dims(S=4, H=2, d_nope=4, d_rope=4, d_v=3, d_kv=6, B=2)
D_MODEL = 5


def _problem(rng, dims, d_model):
    n_h = dims.H
    h = rng.standard_normal((dims.B, dims.S, d_model))
    w_q = rng.standard_normal((d_model, n_h * dims.d_qk)) / math.sqrt(d_model)
    w_kva = rng.standard_normal((d_model, dims.d_kv + dims.d_rope)) / math.sqrt(d_model)
    gamma = 1.0 + 0.1 * rng.standard_normal(dims.d_kv)
    w_kvb = rng.standard_normal((dims.d_kv, n_h * dims.d_head_kv)) / math.sqrt(dims.d_kv)
    w_o = rng.standard_normal((n_h * dims.d_v, d_model)) / math.sqrt(n_h * dims.d_v)
    cos, sin = oracle.rope_tables(dims.S, dims.d_rope)
    dy = rng.standard_normal((dims.B, dims.S, d_model))
    return dict(h=h, w_q=w_q, w_kva=w_kva, gamma=gamma, w_kvb=w_kvb, w_o=w_o), cos, sin, dy


@pytest.mark.parametrize("norm", ["layer", "rms"])
@pytest.mark.parametrize("name", ["h", "w_q", "w_kva", "gamma", "w_kvb", "w_o"])
def test_block_backward_matches_central_differences(name, norm):
    dims = dataclasses.replace(TINY, norm=norm)
    args, cos, sin, dy = _problem(np.random.default_rng(21), dims, D_MODEL)

    def loss():
        y, _ = block_forward(cos=cos, sin=sin, dims=dims, **args)
        return float((y * dy).sum())

    _, st = block_forward(cos=cos, sin=sin, dims=dims, **args)
    g = block_backward(st, dy)
    analytic = {"h": g["dh"], "w_q": g["dw_q"], "w_kva": g["dw_kva"], "gamma": g["dgamma"],
                "w_kvb": g["dw_kvb"], "w_o": g["dw_o"]}[name]
    x = args[name]
    num = np.zeros_like(x)
    eps = 1e-6
    for idx in np.ndindex(x.shape):
        old = x[idx]
        x[idx] = old + eps
        fp = loss()
        x[idx] = old - eps
        fm = loss()
        x[idx] = old
        num[idx] = (fp - fm) / (2 * eps)
    err = np.linalg.norm(analytic - num) / max(np.linalg.norm(num), 1e-30)
    assert err < 1e-7, err


def test_block_with_selection_projections_is_the_per_rank_compute():
    """h = [q_flat | c] and W_q, W_kv_a select those columns, W_o = [I | 0]:
    then y's first n_h*d_v columns are the per-rank output O in head-major
    order, dh = [dq_flat | dc], dW_q / dW_kv_a are h^T dq / h^T dc, and
    dW_kv_b, dgamma equal the per-rank backward's."""
    dims = TINY
    n_h, dq_cols, dc_cols = dims.H, dims.H * dims.d_qk, dims.d_kv + dims.d_rope
    d_model = dq_cols + dc_cols
    rng = np.random.default_rng(5)
    args, cos, sin, dy = _problem(rng, dims, d_model)
    args["w_q"] = np.eye(d_model)[:, :dq_cols]
    args["w_kva"] = np.eye(d_model)[:, dq_cols:]
    args["w_o"] = np.eye(n_h * dims.d_v, d_model)
    h = args["h"]
    y, st = block_forward(cos=cos, sin=sin, dims=dims, **args)
    q = h[..., :dq_cols].reshape(dims.B, dims.S, n_h, dims.d_qk)
    c = h[..., dq_cols:]
    O, _, ost = oracle.forward(q, c, args["w_kvb"], args["gamma"], cos, sin, dims)
    np.testing.assert_allclose(y[..., :n_h * dims.d_v], O.reshape(dims.B, dims.S, -1),
                               rtol=1e-13, atol=1e-13)
    assert np.all(y[..., n_h * dims.d_v:] == 0)
    g = block_backward(st, dy)
    ref = oracle.backward(ost, dy[..., :n_h * dims.d_v].reshape(dims.B, dims.S, n_h, dims.d_v))
    dq_flat = ref["dq"].reshape(dims.B, dims.S, -1)
    np.testing.assert_allclose(g["dh"], np.concatenate([dq_flat, ref["dc"]], -1),
                               rtol=1e-12, atol=1e-12)
    hf = h.reshape(-1, d_model)
    np.testing.assert_allclose(g["dw_q"], hf.T @ dq_flat.reshape(-1, dq_cols), rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(g["dw_kva"], hf.T @ ref["dc"].reshape(-1, dc_cols), rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(g["dw_kvb"], ref["dw"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dgamma"], ref["dgamma"], rtol=1e-12, atol=1e-12)
