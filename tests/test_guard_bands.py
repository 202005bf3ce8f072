"""Out-of-bounds write checks in place of a memory-checker run.

Every output (O, LSE, dq, dc, dW, dgamma) and both workspaces of a call live
inside a larger device buffer, between two 4 KiB bands of a fixed byte
pattern.  After laga_fwd + laga_bwd the bands must be unchanged (a store past
either end of any buffer, e.g. in a ragged tail tile, would change them),
the inputs must be bitwise unchanged, and the outputs must still match the
fp64 oracle.  Lengths cover one token, one short of a tile, one past it and a
ragged multi-tile case, with B = 2 and a shard inside a wider W_kv_b; the
tiny fp32 workload and a non-canonical bf16 shape take the padded path.
"""

import numpy as np
import pytest
import torch

from _harness import check_forward, check_grads, oracle_run
from laga_inputs import config, make_inputs

pytestmark = pytest.mark.gpu

BAND = 4096
PATTERN = torch.tensor([0xA5, 0x5A, 0xC3, 0x3C], dtype=torch.uint8)


class Guarded:
    """One device allocation: [band | payload | band]."""

    def __init__(self, nbytes, dev):
        self.nbytes = nbytes
        self.raw = torch.empty(2 * BAND + nbytes, dtype=torch.uint8, device=dev)
        reps = (self.raw.numel() + 3) // 4
        self.raw.copy_(PATTERN.repeat(reps)[:self.raw.numel()].to(dev))
        self.fill = self.raw.clone()

    def tensor(self, shape, dtype):
        t = self.raw[BAND:BAND + self.nbytes].view(dtype)
        return t.view(*shape)

    def ptr(self):
        return self.raw.data_ptr() + BAND

    def bands_intact(self):
        n = self.raw.numel()
        head = torch.equal(self.raw[:BAND], self.fill[:BAND])
        tail = torch.equal(self.raw[n - BAND:], self.fill[n - BAND:])
        return head, tail


def _nbytes(shape, dtype):
    return int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()


def run_guarded(wl, form):
    import sequence_latent_norm_gb300 as pkg
    lib = pkg._lib
    dev = torch.device("cuda:0")
    cpu = make_inputs(wl)
    t = {k: v.to(dev) for k, v in cpu.items()}
    before = {k: v.clone() for k, v in t.items()}
    dims = lib.make_dims(wl.S, wl.H, B=wl.B, n_h_total=wl.n_h_total, head_offset=wl.head_offset,
                         d_nope=wl.d_nope, d_rope=wl.d_rope, d_v=wl.d_v, d_kv=wl.d_kv,
                         io_dtype=wl.dtype, form=form)
    io, f32 = wl.torch_dtype, torch.float32
    B, S, H = wl.B, wl.S, wl.H
    shapes = dict(O=((B, S, H, wl.d_v), io), LSE=((B, H, S), f32),
                  dq=((B, S, H, wl.d_qk), io), dc=((B, S, wl.d_kv + wl.d_rope), f32),
                  dw=((wl.d_kv, H * (wl.d_nope + wl.d_v)), f32), dgamma=((wl.d_kv,), f32))
    g = {k: Guarded(_nbytes(*v), dev) for k, v in shapes.items()}
    saved = lib.workspace_bytes(dims, lib.WS_SAVED)
    bwd = lib.workspace_bytes(dims, lib.WS_BWD)
    fwd = lib.workspace_bytes(dims, lib.WS_FWD)
    g["ws_saved"], g["ws_bwd"] = Guarded(saved, dev), Guarded(bwd, dev)
    if fwd:
        g["ws_fwd"] = Guarded(fwd, dev)
    st = torch.cuda.current_stream().cuda_stream
    P = {k: v.data_ptr() for k, v in t.items()}
    lib.fwd_scratch(dims, P["q"], P["c"], P["w"], P["gamma"], P["cos"], P["sin"], g["O"].ptr(),
                    g["LSE"].ptr(), g["ws_saved"].ptr(), saved,
                    g["ws_fwd"].ptr() if fwd else 0, fwd, st)
    lib.bwd(dims, P["q"], P["c"], P["w"], P["gamma"], P["cos"], P["sin"], g["O"].ptr(),
            g["LSE"].ptr(), P["dO"], g["dq"].ptr(), g["dc"].ptr(), g["dw"].ptr(),
            g["dgamma"].ptr(), g["ws_saved"].ptr(), saved, g["ws_bwd"].ptr(), bwd, st)
    lib.sync_check()
    for k, gb in g.items():
        head, tail = gb.bands_intact()
        assert head and tail, f"{form} {wl}: band {'before' if not head else 'after'} {k} changed"
    for k in t:
        assert torch.equal(t[k], before[k]), f"{form}: input {k} changed"
    out = {k: g[k].tensor(*shapes[k]).cpu() for k in shapes}
    return cpu, out


CASES = [
    dict(S=1, H=2, B=2, n_h_total=5, head_offset=2),
    dict(S=127, H=2, B=2, n_h_total=5, head_offset=2),
    dict(S=129, H=2, B=2, n_h_total=5, head_offset=3),
    dict(S=333, H=3, B=2, n_h_total=7, head_offset=4),
]


@pytest.mark.parametrize("form", ["laga", "explicit", "absorbed", "laga_fused"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c['S']}")
def test_guard_bands_v3_dims(case, form):
    wl = config(1, **case)
    cpu, got = run_guarded(wl, form)
    ref = oracle_run(wl, cpu)
    check_forward(got, ref, f"{form} {case}", form=form)
    check_grads(got, ref, where=f"{form} {case}")


@pytest.mark.parametrize("form", ["laga", "absorbed", "laga_fused"])
@pytest.mark.parametrize("wl", [config(0), config(1, S=129, H=2, B=2, d_nope=64, d_rope=32,
                                                   d_v=64, d_kv=256)],
                         ids=["fp32-config0", "bf16-small-dims"])
def test_guard_bands_padded_path(wl, form):
    cpu, got = run_guarded(wl, form)
    ref = oracle_run(wl, cpu)
    check_forward(got, ref, f"{form} {wl.name}", form=form)
    check_grads(got, ref, where=f"{form} {wl.name}")
