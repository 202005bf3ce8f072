"""Host-side tests of the C ABI: the library loads, exports every declared
entry point, plans workspaces and rejects bad arguments before any launch."""

import ctypes
import os
import re

import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sequence_latent_norm_gb300.build import build_library
    build_library()
    import sequence_latent_norm_gb300 as pkg
    return pkg._lib


def _declared(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(laga_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared("laga.h")
    assert "laga_fwd" in names and "laga_bwd" in names
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n
    assert set(names) <= set(lib.EXPORTED) | set(names)


def test_workspace_plan_and_tensor_listing(lib):
    d = lib.make_dims(16384, 16)
    saved = lib.workspace_bytes(d, lib.WS_SAVED)
    bwd = lib.workspace_bytes(d, lib.WS_BWD)
    assert saved > 0 and bwd > 0
    ts = lib.workspace_tensors(d, lib.WS_SAVED)
    names = [t[0] for t in ts]
    assert "kv" in names and "L" in names and "q_absorbed" not in names
    for (_, off, nb), (_, off2, _) in zip(ts, ts[1:]):
        assert off + nb <= off2 and off2 % 1024 == 0
    assert ts[-1][1] + ts[-1][2] <= saved
    assert lib.workspace_bytes(lib.make_dims(16384, 16, d_rope=63), lib.WS_SAVED) == 0
    assert lib.workspace_bytes(lib.make_dims(0, 16), lib.WS_SAVED) == 0


def test_backward_scratch_listing_and_dw_split_partials(lib):
    """The backward scratch is laid out like the saved workspace (ordered,
    1024-aligned, inside the reported size); the dW token-split partials, when
    present, are a whole number (2..8) of the shard's fp32 dW."""
    for S, H, B in [(16384, 16, 1), (2048, 8, 1), (4096, 128, 1), (129, 3, 2), (1, 1, 1)]:
        d = lib.make_dims(S, H, B=B)
        bwd = lib.workspace_bytes(d, lib.WS_BWD)
        ts = lib.workspace_tensors(d, lib.WS_BWD)
        assert bwd > 0 and ts
        for (_, off, nb), (_, off2, _) in zip(ts, ts[1:]):
            assert off + nb <= off2 and off2 % 1024 == 0
        assert ts[-1][1] + ts[-1][2] <= bwd
        sizes = dict((n, b) for n, _, b in ts)
        dw_shard = 512 * H * 256 * 4
        if "dw_split_partials" in sizes:
            k, rem = divmod(sizes["dw_split_partials"], dw_shard)
            assert rem == 0 and 2 <= k <= 8, (S, H, B, k)


def test_absorbed_minus_laga_saved_bytes_equal_closed_form(lib):
    """The form-specific activations differ by the pages' mechanism: two
    n_h*d_kv intermediates per token (absorbed) versus per-head K/V (LAGA)."""
    for S, H in [(2048, 8), (16384, 16), (32768, 32)]:
        la = dict((n, b) for n, _, b in lib.workspace_tensors(lib.make_dims(S, H), lib.WS_SAVED))
        ab = dict((n, b) for n, _, b in
                  lib.workspace_tensors(lib.make_dims(S, H, form="absorbed"), lib.WS_SAVED))
        diff = (ab["q_absorbed"] + ab["o_latent"]) - la["kv"]
        assert diff == oracle.activation_bytes("absorbed", S, H) - oracle.activation_bytes("laga", S, H)
        common = set(la) & set(ab)
        assert all(la[n] == ab[n] for n in common)


def _fake(addr):
    return ctypes.c_void_p(addr)


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only safe without a GPU")
def test_bad_arguments_return_status_without_launch(lib):
    so = lib.load()
    d = lib.make_dims(256, 2)
    nb = lib.workspace_bytes(d, lib.WS_SAVED)
    p = [0x10000 * (i + 1) for i in range(9)]

    def fwd(dims, ptrs, ws_bytes=nb):
        return so.laga_fwd(ctypes.byref(dims), *ptrs[:8], ptrs[8], ws_bytes, None)

    assert fwd(d, [0] + p[1:]) == lib.LAGA_ERR_ARG
    assert fwd(d, [p[0] + 8] + p[1:]) == lib.LAGA_ERR_ALIGN
    assert fwd(d, p, nb - 1) == lib.LAGA_ERR_WORKSPACE
    assert fwd(lib.make_dims(256, 2, causal=0), p) == lib.LAGA_ERR_UNSUPPORTED
    assert fwd(lib.make_dims(256, 2, d_nope=24), p) == lib.LAGA_ERR_ARG
    assert fwd(lib.make_dims(256, 2, n_h_total=2, head_offset=1), p) == lib.LAGA_ERR_ARG
    # valid arguments on a machine without a GPU fail in CUDA, not in a crash
    assert fwd(d, p) == lib.LAGA_ERR_CUDA
    assert lib.status_string(lib.LAGA_ERR_TIMEOUT) == "device wait timed out"


def test_noalloc_rejects_latent_wider_than_its_scratch(lib):
    """laga_norm_rope_bwd_noalloc's fixed scratch holds d_kv <= 512 columns;
    a wider latent is refused on the host, before any CUDA call."""
    so = lib.load()
    d = lib.make_dims(128, 2, d_kv=1024)
    null = ctypes.c_void_p(0)
    st = so.laga_norm_rope_bwd_noalloc(ctypes.byref(d), null, null, null, null, null, null,
                                       null, null, null)
    assert st == lib.LAGA_ERR_WORKSPACE
    assert "workspace" in lib.status_string(st)


def test_latent_norm_field_is_validated(lib):
    """dims.norm selects the latent norm (0 LayerNorm, 1 its RMS variant);
    any other value is refused by the plan, before any launch."""
    assert lib.workspace_bytes(lib.make_dims(256, 2, norm="rms"), lib.WS_SAVED) == \
        lib.workspace_bytes(lib.make_dims(256, 2), lib.WS_SAVED)
    d = lib.make_dims(256, 2)
    d.norm = 2
    assert lib.workspace_bytes(d, lib.WS_SAVED) == 0


def test_fused_form_moves_kv_from_saved_to_scratch(lib):
    """The fused form (up-projection rebuilt inside the key-stationary
    backward) keeps no per-head K/V between the passes: the saved workspace
    loses exactly the B*S*H*256 bf16 "kv" tensor, which becomes the forward's
    scratch, and the backward scratch gains one of the same size for the
    rebuilt tiles.  Every other tensor is unchanged."""
    for S, H, B in [(16384, 16, 1), (129, 3, 2), (32768, 32, 1)]:
        la = lib.make_dims(S, H, B=B)
        fu = lib.make_dims(S, H, B=B, form="laga_fused")
        sv_la = dict((n, b) for n, _, b in lib.workspace_tensors(la, lib.WS_SAVED))
        sv_fu = dict((n, b) for n, _, b in lib.workspace_tensors(fu, lib.WS_SAVED))
        kv = B * S * H * 256 * 2
        assert sv_la["kv"] == kv and "kv" not in sv_fu
        assert sv_fu == {n: b for n, b in sv_la.items() if n != "kv"}
        assert lib.workspace_tensors(fu, lib.WS_FWD) == [("kv", 0, kv)]
        assert lib.workspace_bytes(fu, lib.WS_FWD) == kv + (-kv) % 1024
        assert lib.workspace_tensors(la, lib.WS_FWD) == [] and lib.workspace_bytes(la, lib.WS_FWD) == 0
        bw_la = dict((n, b) for n, _, b in lib.workspace_tensors(la, lib.WS_BWD))
        bw_fu = dict((n, b) for n, _, b in lib.workspace_tensors(fu, lib.WS_BWD))
        assert bw_fu.pop("kv_rebuilt") == kv and bw_fu == bw_la
        assert lib.workspace_bytes(la, lib.WS_SAVED) - lib.workspace_bytes(fu, lib.WS_SAVED) >= kv


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only safe without a GPU")
def test_fused_form_forward_needs_its_scratch(lib):
    """laga_fwd (no scratch) refuses the fused form; laga_fwd_scratch checks
    the scratch's size and alignment before any CUDA call."""
    so = lib.load()
    d = lib.make_dims(256, 2, form="laga_fused")
    nb = lib.workspace_bytes(d, lib.WS_SAVED)
    fb = lib.workspace_bytes(d, lib.WS_FWD)
    p = [0x10000 * (i + 1) for i in range(10)]
    assert so.laga_fwd(ctypes.byref(d), *p[:9], nb, None) == lib.LAGA_ERR_WORKSPACE
    fs = so.laga_fwd_scratch
    assert fs(ctypes.byref(d), *p[:9], nb, None, fb, None) == lib.LAGA_ERR_WORKSPACE
    assert fs(ctypes.byref(d), *p[:9], nb, p[9], fb - 1, None) == lib.LAGA_ERR_WORKSPACE
    assert fs(ctypes.byref(d), *p[:9], nb, p[9] + 8, fb, None) == lib.LAGA_ERR_ALIGN
    assert fs(ctypes.byref(d), *p[:9], nb, p[9], fb, None) == lib.LAGA_ERR_CUDA
