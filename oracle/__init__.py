"""Plain fp64 CPU oracle for the per-rank LAGA compute.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code, tables or helpers with the CUDA path in
``sequence_latent_norm_gb300``; the two meet only through the seeded input
generators in ``laga_inputs``.

Every function follows the definitions on the LAGA paper page
("A Training-Memory Regression in MLA Sequence Parallelism ... LAGA",
arXiv 2607.17644v1): Section 2.1 (MLA), Section 3.3 Algorithm 1, Section 5.1
equation for k_nope / v, Section 5.2 (backward and the W_kv_b gradient
shard), Section 5.3 (decoupled RoPE) and Section 3.2 (the absorbed form).
Where the page is silent the reading taken is stated at the function.

Parity status per function (what pins it lives in ``tests/test_oracle.py``):

* ``layernorm``            pinned: torch.nn.functional.layer_norm (fp64),
                           affine-shift invariance, brute-force loops.
* ``rmsnorm``              pinned: torch.nn.functional.rms_norm (fp64),
                           positive-scale invariance, not shift-invariant;
                           its backward by finite differences and autograd.
* ``rope_tables``/``rope`` pinned: position-0 identity, norm preservation,
                           relative-position shift invariance, brute force.
* ``forward``              pinned: brute-force Python loops on tiny inputs,
                           torch SDPA (fp64) on the d_rope=0, W=[I|I] case,
                           q=0 closed form, row-0 closed form, rows of P
                           summing to one.
* ``backward``             pinned: central finite differences of forward,
                           torch autograd (fp64) on the reduced case,
                           sum_j dS_ij = 0, sum over features of dx_LN = 0.
* ``forward_absorbed`` /
  ``backward_absorbed``    pinned: equal to the explicit form to fp64
                           round-off (Propositions 1-2), finite differences.
* ``emulate_sp``           pinned: equal to the unsharded result.
* ``comm_bytes_per_rank``  pinned: every cell of Table 1 and the n_h sweep
                           ratios printed in Section 4.2.
* ``activation_elems``     pinned: the n_h*d_kv versus H*(d_nope+d_v)
                           per-token ratio stated in Sections 1, 3.2, 3.3.
* ``block.block_forward`` /
  ``block.block_backward`` the attention block of Algorithm 1 (W_q, W_kv_a,
                           the per-rank compute, W_o) at one rank; pinned
                           by central finite differences and by selection-
                           matrix projections reducing it to ``forward`` /
                           ``backward`` (tests/test_oracle_block.py).
"""

from .laga import (  # noqa: F401
    Dims,
    layernorm,
    layernorm_backward,
    rmsnorm,
    rmsnorm_backward,
    latent_norm,
    latent_norm_backward,
    rope_tables,
    rope,
    rope_transpose,
    forward,
    backward,
    forward_absorbed,
    backward_absorbed,
    emulate_sp,
    shard_weights,
    comm_bytes_per_rank,
    activation_elems_per_token,
    activation_bytes,
)
