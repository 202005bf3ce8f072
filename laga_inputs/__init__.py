"""Seeded synthetic inputs shared by the oracle checks, the GPU tests and the bench.

This module holds no arithmetic of the method: it draws the input tensors
(q, c, W_kv_b, gamma, dO) and builds the RoPE cos/sin tables that the
boundary takes as inputs.  Distributions follow the workload descriptions:
q ~ N(0,1), c ~ N(0,1), W_kv_b ~ N(0, 1/d_kv) (the second argument read as a
variance), gamma = 1 + N(0, 0.1) (0.1 read as a standard deviation),
dO ~ N(0,1), RoPE theta = 10000.  Every draw comes from a CPU
``torch.Generator`` seeded with ``1000 + config`` in fp32 and is then cast to
the I/O dtype, so the oracle and the GPU path see identical values.

No public dataset is involved: the LAGA page measures on random data and
fixed DeepSeek-V3 dimensions only.
"""

from __future__ import annotations

import dataclasses
import math

import torch

DEEPSEEK_V3 = dict(d_nope=128, d_rope=64, d_v=128, d_kv=512)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    S: int
    H: int                      # heads of the shard this process computes
    n_h_total: int              # heads whose columns W_kv_b holds
    head_offset: int = 0
    d_nope: int = 128
    d_rope: int = 64
    d_v: int = 128
    d_kv: int = 512
    B: int = 1
    dtype: str = "bf16"         # I/O dtype of q, c, W_kv_b, O, dq, dO
    seed: int = 1000
    theta: float = 10000.0
    norm: str = "layer"         # latent norm: "layer" or its RMS variant "rms"

    @property
    def d_qk(self):
        return self.d_nope + self.d_rope

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "fp32": torch.float32}[self.dtype]


def config(k: int, **over) -> Workload:
    """The five workload configurations (sizes of the shard; seed 1000+k)."""
    base = {
        0: dict(name="tiny-mla-fp32", S=128, H=4, n_h_total=4, d_nope=32, d_rope=16,
                d_v=32, d_kv=64, dtype="fp32"),
        1: dict(name="v3-shard16-s4096", S=4096, H=16, n_h_total=16, **DEEPSEEK_V3),
        2: dict(name="v3-shard16-s16384", S=16384, H=16, n_h_total=16, **DEEPSEEK_V3),
        3: dict(name="v3-heads128-s4096", S=4096, H=128, n_h_total=128, **DEEPSEEK_V3),
        4: dict(name="v3-sweep", S=4096, H=16, n_h_total=16, **DEEPSEEK_V3),
    }[k]
    base.update(seed=1000 + k)
    base.update(over)
    return Workload(**base)


def rope_tables(S: int, d_rope: int, theta: float = 10000.0):
    """cos/sin [S, d_rope/2] fp32 for positions 0..S-1 of the gathered sequence."""
    half = d_rope // 2
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d_rope)
    ang = torch.arange(S, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).float().contiguous(), torch.sin(ang).float().contiguous()


def make_inputs(wl: Workload, with_grad_out: bool = True):
    """Draw one workload's inputs on the CPU.

    Returns a dict of CPU tensors: q [B,S,H,d_nope+d_rope], c [B,S,d_kv+d_rope],
    w [d_kv, n_h_total*(d_nope+d_v)] (all in the I/O dtype), gamma [d_kv] fp32,
    cos/sin [S, d_rope/2] fp32 and dO [B,S,H,d_v] (I/O dtype).
    """
    g = torch.Generator(device="cpu").manual_seed(wl.seed)
    dt = wl.torch_dtype
    q = torch.randn(wl.B, wl.S, wl.H, wl.d_qk, generator=g)
    c = torch.randn(wl.B, wl.S, wl.d_kv + wl.d_rope, generator=g)
    w = torch.randn(wl.d_kv, wl.n_h_total * (wl.d_nope + wl.d_v), generator=g) / math.sqrt(wl.d_kv)
    gamma = 1.0 + 0.1 * torch.randn(wl.d_kv, generator=g)
    out = dict(q=q.to(dt).contiguous(), c=c.to(dt).contiguous(), w=w.to(dt).contiguous(),
               gamma=gamma.float().contiguous())
    out["cos"], out["sin"] = rope_tables(wl.S, wl.d_rope, wl.theta)
    if with_grad_out:
        out["dO"] = torch.randn(wl.B, wl.S, wl.H, wl.d_v, generator=g).to(dt).contiguous()
    return out


def as_f64(t: torch.Tensor):
    """The exact values of a tensor as a float64 NumPy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def make_block_inputs(wl: Workload, d_model: int):
    """Draw the inputs of the attention block around one workload (all heads
    at one rank: n_h = wl.H): h [B, S, d_model] ~ N(0, 1); W_q [d_model,
    n_h (d_nope + d_rope)] and W_kv_a [d_model, d_kv + d_rope] ~ N(0,
    1/d_model), so that q and c keep the workload's unit variance; W_kv_b and
    gamma as ``make_inputs``; W_o [n_h d_v, d_model] ~ N(0, 1/(n_h d_v));
    dy [B, S, d_model] ~ N(0, 1).  Matrices in the I/O dtype, gamma and the
    RoPE tables fp32, all on the CPU."""
    g = torch.Generator(device="cpu").manual_seed(wl.seed + 7919)
    dt = wl.torch_dtype
    n_h = wl.H
    h = torch.randn(wl.B, wl.S, d_model, generator=g)
    w_q = torch.randn(d_model, n_h * wl.d_qk, generator=g) / math.sqrt(d_model)
    w_kva = torch.randn(d_model, wl.d_kv + wl.d_rope, generator=g) / math.sqrt(d_model)
    w_kvb = torch.randn(wl.d_kv, n_h * (wl.d_nope + wl.d_v), generator=g) / math.sqrt(wl.d_kv)
    gamma = 1.0 + 0.1 * torch.randn(wl.d_kv, generator=g)
    w_o = torch.randn(n_h * wl.d_v, d_model, generator=g) / math.sqrt(n_h * wl.d_v)
    dy = torch.randn(wl.B, wl.S, d_model, generator=g)
    out = {k: v.to(dt).contiguous() for k, v in
           dict(h=h, w_q=w_q, w_kva=w_kva, w_kvb=w_kvb, w_o=w_o, dy=dy).items()}
    out["gamma"] = gamma.float().contiguous()
    out["cos"], out["sin"] = rope_tables(wl.S, wl.d_rope, wl.theta)
    return out
