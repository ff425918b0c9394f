"""GB300-native block-sparse masked attention (Splash-style): forward and
backward.

The compute runs in libbsm.so (hand-written CUDA for sm_103a) behind the C
ABI of ``include/bsm.h``; this package is its Python binding.
"""

from .api import (  # noqa: F401
    MASK_BAND,
    MASK_CAUSAL,
    MASK_DENSE,
    MASK_LOCAL,
    MASK_SEGMENT,
    SCORE_POINTWISE,
    SCORE_SOFTMAX,
    BsmError,
    MaskInfo,
    bsm_build_mask_info,
    bsm_device_status,
    bsm_last_error,
    bsm_mask_info_bytes,
    bsm_pack_dense_mask,
    bsm_selftest_wait_timeout,
    bsm_splash_bwd,
    bsm_splash_bwd_workspace_bytes,
    bsm_splash_fwd,
    bsm_splash_fwd_host,
    bsm_splash_fwd_host_bytes,
    bsm_splash_fwd_workspace_bytes,
    bsm_version,
    build_mask_info,
    pack_dense_mask,
    splash_attention,
    splash_attention_bwd,
)
