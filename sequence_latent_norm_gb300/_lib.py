"""ctypes binding of liblaga.so: argument marshalling only.

Every step of the compute runs in the library's CUDA kernels; this module
turns Python values into the C structs and pointers of ``include/laga.h``
and raises on a non-OK status.  It never falls back to another
implementation: if the library is missing, loading raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liblaga.so")

LAGA_OK, LAGA_ERR_ARG, LAGA_ERR_ALIGN, LAGA_ERR_WORKSPACE = 0, 1, 2, 3
LAGA_ERR_UNSUPPORTED, LAGA_ERR_CUDA, LAGA_ERR_TIMEOUT = 4, 5, 6
FORMS = {"laga": 0, "explicit": 1, "absorbed": 2, "laga_fused": 3}
DTYPES = {"bf16": 0, "fp32": 1}
NORMS = {"layer": 0, "rms": 1}
WS_SAVED, WS_BWD, WS_FWD = 0, 1, 2

EXPORTED = ("laga_workspace_bytes", "laga_workspace_tensor", "laga_fwd", "laga_fwd_scratch",
            "laga_bwd",
            "laga_bwd_overlap", "laga_sync_check", "laga_status_string", "laga_last_launch_count",
            "laga_profile_enable", "laga_profile_reset", "laga_profile_read",
            "laga_norm_rope_bwd_noalloc", "laga_selftest_wait_timeout", "laga_diag_mma_rate")


class LagaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("S", ctypes.c_int), ("n_h_total", ctypes.c_int),
                ("head_offset", ctypes.c_int), ("n_h_shard", ctypes.c_int),
                ("d_nope", ctypes.c_int), ("d_rope", ctypes.c_int), ("d_v", ctypes.c_int),
                ("d_kv", ctypes.c_int), ("scale", ctypes.c_float), ("ln_eps", ctypes.c_float),
                ("causal", ctypes.c_int), ("io_dtype", ctypes.c_int), ("form", ctypes.c_int),
                ("norm", ctypes.c_int)]


class LagaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library once (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"liblaga.so not found at {path}: build it with "
                           "sequence_latent_norm_gb300.build.build_library()")
    lib = ctypes.CDLL(path)
    P, S, I, F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_float)
    D = ctypes.POINTER(LagaDims)
    lib.laga_workspace_bytes.argtypes = [D, I]
    lib.laga_workspace_bytes.restype = S
    lib.laga_workspace_tensor.argtypes = [D, I, I, ctypes.POINTER(ctypes.c_char_p),
                                          ctypes.POINTER(S), ctypes.POINTER(S)]
    lib.laga_workspace_tensor.restype = I
    lib.laga_fwd.argtypes = [D, P, P, P, P, P, P, P, P, P, S, P]
    lib.laga_fwd.restype = I
    lib.laga_fwd_scratch.argtypes = [D, P, P, P, P, P, P, P, P, P, S, P, S, P]
    lib.laga_fwd_scratch.restype = I
    lib.laga_bwd.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P, S, P]
    lib.laga_bwd.restype = I
    lib.laga_bwd_overlap.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P, S, P,
                                     P, P, P]
    lib.laga_bwd_overlap.restype = I
    lib.laga_sync_check.argtypes = [P]
    lib.laga_sync_check.restype = I
    lib.laga_selftest_wait_timeout.argtypes = [P]
    lib.laga_selftest_wait_timeout.restype = I
    lib.laga_status_string.argtypes = [I]
    lib.laga_status_string.restype = ctypes.c_char_p
    lib.laga_last_launch_count.argtypes = []
    lib.laga_last_launch_count.restype = I
    lib.laga_profile_enable.argtypes = [I]
    lib.laga_profile_enable.restype = None
    lib.laga_profile_reset.argtypes = []
    lib.laga_profile_reset.restype = None
    lib.laga_profile_read.argtypes = [ctypes.POINTER(ctypes.c_char_p),
                                      ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I), I]
    lib.laga_profile_read.restype = I
    lib.laga_norm_rope_bwd_noalloc.argtypes = [D, P, P, P, P, P, P, P, P, P]
    lib.laga_norm_rope_bwd_noalloc.restype = I
    lib.laga_diag_mma_rate.argtypes = [I, I, I, I, I, I, P, P]
    lib.laga_diag_mma_rate.restype = I
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().laga_status_string(int(status)).decode()


def make_dims(S, n_h_shard, *, B=1, n_h_total=None, head_offset=0, d_nope=128, d_rope=64,
              d_v=128, d_kv=512, scale=0.0, ln_eps=1e-5, causal=1, io_dtype="bf16",
              form="laga", norm="layer") -> LagaDims:
    return LagaDims(B, S, n_h_shard if n_h_total is None else n_h_total, head_offset, n_h_shard,
                    d_nope, d_rope, d_v, d_kv, scale, ln_eps, causal, DTYPES[io_dtype],
                    FORMS[form], NORMS[norm])


def workspace_bytes(dims: LagaDims, pass_: int) -> int:
    return int(load().laga_workspace_bytes(ctypes.byref(dims), pass_))


def workspace_tensors(dims: LagaDims, pass_: int):
    """[(name, offset, bytes)] of the tensors inside one workspace."""
    lib = load()
    out, i = [], 0
    name, off, nb = ctypes.c_char_p(), ctypes.c_size_t(), ctypes.c_size_t()
    while lib.laga_workspace_tensor(ctypes.byref(dims), pass_, i, ctypes.byref(name),
                                    ctypes.byref(off), ctypes.byref(nb)) == LAGA_OK:
        out.append((name.value.decode(), off.value, nb.value))
        i += 1
    return out


def _check(status: int, what: str):
    if status != LAGA_OK:
        raise LagaError(status, what)


def fwd(dims: LagaDims, q, c, w, gamma, cos, sin, o, lse, ws_saved, saved_bytes, stream=0):
    """laga_fwd with raw device addresses (ints)."""
    _check(load().laga_fwd(ctypes.byref(dims), q, c, w, gamma, cos, sin, o, lse, ws_saved,
                           saved_bytes, stream), "laga_fwd")


def fwd_scratch(dims: LagaDims, q, c, w, gamma, cos, sin, o, lse, ws_saved, saved_bytes, ws_fwd,
                fwd_bytes, stream=0):
    """laga_fwd_scratch with raw device addresses (ints)."""
    _check(load().laga_fwd_scratch(ctypes.byref(dims), q, c, w, gamma, cos, sin, o, lse, ws_saved,
                                   saved_bytes, ws_fwd, fwd_bytes, stream), "laga_fwd_scratch")


def bwd(dims: LagaDims, q, c, w, gamma, cos, sin, o, lse, d_o, dq, dc, dw, dgamma, ws_saved,
        saved_bytes, ws_bwd, bwd_bytes, stream=0):
    """laga_bwd with raw device addresses (ints)."""
    _check(load().laga_bwd(ctypes.byref(dims), q, c, w, gamma, cos, sin, o, lse, d_o, dq, dc, dw,
                           dgamma, ws_saved, saved_bytes, ws_bwd, bwd_bytes, stream), "laga_bwd")


def bwd_overlap(dims: LagaDims, q, c, w, gamma, cos, sin, o, lse, d_o, dq, dc, dw, dgamma,
                ws_saved, saved_bytes, ws_bwd, bwd_bytes, stream, aux_stream, fork_event,
                join_event):
    """laga_bwd_overlap with raw device addresses and stream/event handles (ints)."""
    _check(load().laga_bwd_overlap(ctypes.byref(dims), q, c, w, gamma, cos, sin, o, lse, d_o, dq,
                                   dc, dw, dgamma, ws_saved, saved_bytes, ws_bwd, bwd_bytes,
                                   stream, aux_stream, fork_event, join_event),
           "laga_bwd_overlap")


def sync_check(stream=0):
    _check(load().laga_sync_check(stream), "laga_sync_check")


def selftest_wait_timeout(stream=0):
    """Enqueue the bounded-wait self-test (see include/laga.h)."""
    _check(load().laga_selftest_wait_timeout(stream), "laga_selftest_wait_timeout")


def last_launch_count() -> int:
    return int(load().laga_last_launch_count())


def profile_enable(on: bool):
    load().laga_profile_enable(1 if on else 0)


def profile_reset():
    load().laga_profile_reset()


def profile_read():
    """{kernel name: (total ms, launches)} since the last reset (waits for the events)."""
    lib = load()
    n = 64
    names = (ctypes.c_char_p * n)()
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    k = lib.laga_profile_read(names, ms, cnt, n)
    return {names[i].decode(): (ms[i], cnt[i]) for i in range(min(k, n))}


def norm_rope_bwd_noalloc(dims: LagaDims, c, gamma, cos, sin, d_latent, d_kpe_rot, dc, dgamma,
                          stream=0):
    """laga_norm_rope_bwd_noalloc with raw device addresses (ints): the
    LayerNorm + RoPE backward using the library's own fixed scratch."""
    _check(load().laga_norm_rope_bwd_noalloc(ctypes.byref(dims), c, gamma, cos, sin, d_latent,
                                             d_kpe_rot, dc, dgamma, stream),
           "laga_norm_rope_bwd_noalloc")


def diag_mma_rate(form: int, n: int, n_acc: int, run: int, n_instr: int, n_cta: int, cycles,
                  stream=0):
    """laga_diag_mma_rate: SM clocks per CTA for n_instr MMAs into `cycles`
    (a device address of n_cta uint64)."""
    _check(load().laga_diag_mma_rate(form, n, n_acc, run, n_instr, n_cta, cycles, stream),
           "laga_diag_mma_rate")
