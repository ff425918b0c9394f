"""The forward entry point that allocates nothing, called through the C ABI.

bsm_splash_fwd_noalloc serves callers that cannot allocate device memory
(plugins handed finished buffers, engines that reserve all HBM up front,
loops that cannot afford cudaMalloc's synchronisation): its workspace is a
static device array inside the library.  Its output must match the regular
entry point's (which takes a caller-allocated workspace) on two calls in a
row, so the array's state left by one call does not affect the next.  This
file is collected last so that a failure here leaves every other test run.
"""

import ctypes

import numpy as np
import pytest
import torch

import block_sparse_masked_build_gb300 as bsm
from block_sparse_masked_build_gb300 import _lib
from block_sparse_masked_build_gb300 import workloads as wl
from block_sparse_masked_build_gb300._lib import I64x3
from gpu_helpers import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu


def _strides(t):
    return I64x3(t.stride(0), t.stride(1), t.stride(2))


def _noalloc(q, k, v, info, seg, scale, score, out, lse):
    B, H, Sq, D = q.shape
    st = _lib.lib().bsm_splash_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides(q), _strides(k),
        _strides(v), _strides(out), B, H, k.shape[1], Sq, k.shape[2], D,
        ctypes.byref(info.struct), None if seg is None else seg.data_ptr(),
        None if seg is None else seg.data_ptr(), ctypes.c_float(scale), score,
        out.data_ptr(), None if lse is None else lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, _lib.last_error()


@pytest.mark.parametrize("score", [bsm.SCORE_SOFTMAX, bsm.SCORE_POINTWISE])
def test_noalloc_matches_workspace_entry_point(score):
    dev = torch.device("cuda")
    B, H, S, D = 2, 4, 1536, 128
    g = torch.Generator().manual_seed(31)
    q, k, v = (torch.randn(B, H, S, D, generator=g).to(torch.bfloat16).to(dev)
               for _ in range(3))
    seg = torch.from_numpy(wl.random_segment_ids(B, S, 50, 700, 8)).to(dev)
    flags = bsm.MASK_CAUSAL | bsm.MASK_SEGMENT
    info = bsm.build_mask_info(flags, B, S, S, 128, 128, 0, seg, seg,
                               device=dev)
    scale = 0.08
    ref = torch.empty(B, H, S, D, dtype=torch.bfloat16, device=dev)
    ref_lse = torch.empty(B, H, S, device=dev) \
        if score == bsm.SCORE_SOFTMAX else None
    bsm.bsm_splash_fwd(q, k, v, info, seg, seg, scale, score, ref, ref_lse)
    torch.cuda.synchronize()
    scale_ref = float(ref.float().abs().max())
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan")) \
            if ref_lse is not None else None
        _noalloc(q, k, v, info, seg, scale, score, out, lse)
        torch.cuda.synchronize()
        assert bsm.bsm_device_status()[0] == 0
        err = (out.float() - ref.float()).abs()
        if score == bsm.SCORE_POINTWISE:  # outputs ~1e-3: scale the gates
            err = err / scale_ref
        assert torch.isfinite(out.float()).all(), f"call {call}"
        assert err.max().item() <= MAX_ABS, f"call {call}"
        assert err.mean().item() <= MEAN_ABS, f"call {call}"
        if lse is not None:
            rel = (lse - ref_lse).abs() / ref_lse.abs().clamp_min(1.0)
            assert rel.max().item() <= 1e-3, f"call {call}"
