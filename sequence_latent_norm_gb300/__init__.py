"""GB300 (sm_103a) per-rank compute of LAGA (Latent All-Gather Attention).

After the latent all-gather, one rank normalises the gathered MLA latent,
rebuilds its head shard of K/V with the kv_b up-projection and runs causal
MLA attention forward and backward.  All of it runs in the hand-written CUDA
kernels of ``liblaga.so`` (C ABI in ``include/laga.h``); this package is the
build script and a thin binding.
"""

from .api import Laga, Shard, attention_flops, upproj_flops  # noqa: F401
from . import _lib  # noqa: F401
from ._lib import LagaError, WS_BWD, WS_SAVED  # noqa: F401
