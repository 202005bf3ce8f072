"""Torch-tensor front end of the C ABI.

PyTorch supplies device memory and the stream; the binding checks that each
tensor has the shape, dtype, device and contiguity the C ABI assumes (the
C side only sees pointers) and passes the addresses through.
"""

from __future__ import annotations

import dataclasses

import torch

from . import _lib

_TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


@dataclasses.dataclass
class Shard:
    """One rank's problem: sizes of the head shard and the form to run."""

    S: int
    H: int
    n_h_total: int | None = None
    head_offset: int = 0
    B: int = 1
    d_nope: int = 128
    d_rope: int = 64
    d_v: int = 128
    d_kv: int = 512
    scale: float = 0.0
    ln_eps: float = 1e-5
    io_dtype: str = "bf16"
    form: str = "laga"       # "laga", "laga_fused", "explicit" or "absorbed"
    norm: str = "layer"      # latent norm: "layer" (LayerNorm) or "rms" (its RMS variant)

    def dims(self) -> _lib.LagaDims:
        return _lib.make_dims(self.S, self.H, B=self.B, n_h_total=self.n_h_total,
                              head_offset=self.head_offset, d_nope=self.d_nope,
                              d_rope=self.d_rope, d_v=self.d_v, d_kv=self.d_kv, scale=self.scale,
                              ln_eps=self.ln_eps, io_dtype=self.io_dtype, form=self.form,
                              norm=self.norm)

    @property
    def n_total(self):
        return self.H if self.n_h_total is None else self.n_h_total

    @property
    def dtype(self):
        return _TORCH_DT[self.io_dtype]


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, shape, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype} != {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class Laga:
    """Owns the two workspaces of one shard and runs laga_fwd / laga_bwd."""

    def __init__(self, shard: Shard, device="cuda"):
        self.shard = shard
        self.device = torch.device(device)
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.c_dims = shard.dims()
        self.saved_bytes = _lib.workspace_bytes(self.c_dims, _lib.WS_SAVED)
        self.bwd_bytes = _lib.workspace_bytes(self.c_dims, _lib.WS_BWD)
        self.fwd_bytes = _lib.workspace_bytes(self.c_dims, _lib.WS_FWD)
        if self.saved_bytes == 0:
            raise ValueError(f"invalid shard dims {shard}")
        self.ws_saved = torch.empty(self.saved_bytes, dtype=torch.uint8, device=self.device)
        self._ws_bwd = None

    @property
    def ws_bwd(self):
        if self._ws_bwd is None:
            self._ws_bwd = torch.empty(self.bwd_bytes, dtype=torch.uint8, device=self.device)
        return self._ws_bwd

    def _shapes(self):
        s = self.shard
        return dict(q=(s.B, s.S, s.H, s.d_nope + s.d_rope), c=(s.B, s.S, s.d_kv + s.d_rope),
                    w=(s.d_kv, s.n_total * (s.d_nope + s.d_v)), gamma=(s.d_kv,),
                    cos=(s.S, s.d_rope // 2), sin=(s.S, s.d_rope // 2),
                    o=(s.B, s.S, s.H, s.d_v), lse=(s.B, s.H, s.S),
                    dq=(s.B, s.S, s.H, s.d_nope + s.d_rope), dc=(s.B, s.S, s.d_kv + s.d_rope),
                    dw=(s.d_kv, s.H * (s.d_nope + s.d_v)), dgamma=(s.d_kv,))

    def _ptrs(self, **tensors):
        shp, dt, f32 = self._shapes(), self.shard.dtype, torch.float32
        io = {"q", "c", "w", "o", "dO", "dq"}
        out = {}
        for k, t in tensors.items():
            key = "o" if k == "dO" else k
            out[k] = _need(t, k, shp[key], dt if k in io else f32, self.device)
        return out

    def forward(self, q, c, w, gamma, cos, sin, o=None, lse=None, stream=None):
        s = self.shard
        shp = self._shapes()
        if o is None:
            o = torch.empty(shp["o"], dtype=s.dtype, device=self.device)
        if lse is None:
            lse = torch.empty(shp["lse"], dtype=torch.float32, device=self.device)
        p = self._ptrs(q=q, c=c, w=w, gamma=gamma, cos=cos, sin=sin, o=o, lse=lse)
        # the forward scratch (the fused form's K/V) is released on return:
        # the caching allocator hands it out again only in stream order
        scratch = (torch.empty(self.fwd_bytes, dtype=torch.uint8, device=self.device)
                   if self.fwd_bytes else None)
        if scratch is not None and stream is not None:
            scratch.record_stream(stream)
        _lib.fwd_scratch(self.c_dims, p["q"], p["c"], p["w"], p["gamma"], p["cos"], p["sin"],
                         p["o"], p["lse"], self.ws_saved.data_ptr(), self.saved_bytes,
                         scratch.data_ptr() if scratch is not None else 0, self.fwd_bytes,
                         _stream_handle(stream))
        return o, lse

    def _overlap_events(self):
        """Two events of this object for laga_bwd_overlap (created by a first
        record, so that their handles exist)."""
        if getattr(self, "_events", None) is None:
            evs = (torch.cuda.Event(), torch.cuda.Event())
            with torch.cuda.device(self.device):
                for e in evs:
                    e.record(torch.cuda.current_stream(self.device))
            self._events = evs
        return self._events

    def backward(self, q, c, w, gamma, cos, sin, o, lse, dO, dq=None, dc=None, dw=None,
                 dgamma=None, stream=None, aux_stream=None):
        """laga_bwd; with ``aux_stream`` (a torch.cuda.Stream other than the
        compute stream) laga_bwd_overlap, which runs the dQ kernel there."""
        s = self.shard
        shp = self._shapes()
        f32 = torch.float32
        dq = torch.empty(shp["dq"], dtype=s.dtype, device=self.device) if dq is None else dq
        dc = torch.empty(shp["dc"], dtype=f32, device=self.device) if dc is None else dc
        dw = torch.empty(shp["dw"], dtype=f32, device=self.device) if dw is None else dw
        dgamma = torch.empty(shp["dgamma"], dtype=f32, device=self.device) if dgamma is None else dgamma
        p = self._ptrs(q=q, c=c, w=w, gamma=gamma, cos=cos, sin=sin, o=o, lse=lse, dO=dO, dq=dq,
                       dc=dc, dw=dw, dgamma=dgamma)
        args = (self.c_dims, p["q"], p["c"], p["w"], p["gamma"], p["cos"], p["sin"], p["o"],
                p["lse"], p["dO"], p["dq"], p["dc"], p["dw"], p["dgamma"],
                self.ws_saved.data_ptr(), self.saved_bytes, self.ws_bwd.data_ptr(),
                self.bwd_bytes, _stream_handle(stream))
        if aux_stream is None:
            _lib.bwd(*args)
        else:
            fork, join = self._overlap_events()
            _lib.bwd_overlap(*args, aux_stream.cuda_stream, fork.cuda_event, join.cuda_event)
        return dq, dc, dw, dgamma

    def workspace_tensors(self, pass_):
        return _lib.workspace_tensors(self.c_dims, pass_)


def attention_flops(S: int, H: int, d_qk: int = 192, d_v: int = 128, B: int = 1):
    """Algorithmic FLOPs of causal attention, counting S^2/2 query-key pairs.

    Forward per pair: 2 d_qk (scores) + 2 d_v (P V).  Backward per pair:
    2 d_qk (score recompute) + 2 d_v (dP) + 2 d_v (dV) + 2 d_qk (dK) +
    2 d_qk (dQ).  Returns (fwd, bwd).
    """
    pairs = B * H * S * S / 2.0
    return pairs * (2 * d_qk + 2 * d_v), pairs * (6 * d_qk + 4 * d_v)


def upproj_flops(S: int, H: int, d_kv: int = 512, d_head: int = 256, B: int = 1):
    """FLOPs of the up-projection forward and of its two backward GEMMs."""
    f = 2.0 * B * S * d_kv * H * d_head
    return f, 2 * f
