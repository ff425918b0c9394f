"""fp64 CPU oracle for block-sparse masked attention -- TEST INFRASTRUCTURE ONLY.

Nothing in the product path may import, call or execute this package.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs
of ``bench.py`` use it.  It shares no code with the CUDA path: it is a plain,
slow, obviously-correct restatement of what the forward pass computes,
written from the pages it cites:

* "Splash Attention" notes ("JAX 到 VLIW, Pallas / Splash Attention 复习笔记"),
  section 12 (naive attention), section 15 (online softmax m/l/o), section 21
  (sparse K/V indirection through ``data_next``);
* RecML ``recml/core/ops/hstu_ops.py`` (pointwise HSTU splash attention):
  ``_next_nonzero`` (block classes 0/1/2), ``_apply_mask`` (per-element mask),
  ``_pointwise_splash_attention_fwd_kernel_impl`` (pointwise score path),
  ``pointwise_splash_attention`` (defaults and argument checks).

Every function is pinned by ``tests/test_oracle_pins.py`` and
``tests/test_oracle_mask_info.py`` against facts that do not come from the
oracle itself (closed forms, a worked example printed in the pages, library
special cases, invariants).
"""

from .splash_oracle import (  # noqa: F401
    MASK_BAND,
    MASK_CAUSAL,
    MASK_DENSE,
    MASK_LOCAL,
    MASK_SEGMENT,
    visible,
    visibility_matrix,
    mask_info,
    visible_pair_count,
    softmax_attention,
    softmax_attention_online,
    pointwise_attention,
    softmax_attention_bwd,
    pointwise_attention_bwd,
    unmasked_flops,
)
