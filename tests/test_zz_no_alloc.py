"""The forward entry point that allocates nothing, called through the C ABI.

bsm_splash_fwd_noalloc serves callers that cannot allocate device memory
(plugins handed finished buffers, engines that reserve all HBM up front,
loops that cannot afford cudaMalloc's synchronisation): its workspace is a
static device array inside the library.  It runs the same kernel as the
regular entry point (which takes a caller-allocated workspace), with the
same deterministic schedule, so its outputs must be bit-identical to that
entry point's, on two calls in a row, and after a larger problem has left
its state in the shared array.  After its first call in a context, a call
takes no device memory.  This file is collected last so that a failure here
leaves every other test run.
"""

import ctypes

import pytest
import torch

import block_sparse_masked_build_gb300 as bsm
from block_sparse_masked_build_gb300 import _lib
from block_sparse_masked_build_gb300 import workloads as wl
from block_sparse_masked_build_gb300._lib import I64x3

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


def _problem(B, H, S, D, seed, segmented):
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(B, H, S, D, generator=g).to(torch.bfloat16).to(dev)
               for _ in range(3))
    seg = None
    flags = bsm.MASK_CAUSAL
    if segmented:
        seg = torch.from_numpy(
            wl.random_segment_ids(B, S, 50, 700, seed + 1)).to(dev)
        flags |= bsm.MASK_SEGMENT
    info = bsm.build_mask_info(flags, B, S, S, 128, 128, 0, seg, seg,
                               device=dev)
    return q, k, v, seg, info


@pytest.mark.parametrize("score", [bsm.SCORE_SOFTMAX, bsm.SCORE_POINTWISE])
def test_noalloc_matches_workspace_entry_point(score):
    # a larger problem first (more units, longer lists), then a smaller one:
    # whatever the first leaves in the shared array must not leak into the
    # second
    scale = 0.08
    for (B, H, S, D, seed, segmented) in [(2, 8, 4096, 128, 31, False),
                                          (2, 4, 1536, 128, 41, True),
                                          (1, 2, 640, 64, 51, True)]:
        q, k, v, seg, info = _problem(B, H, S, D, seed, segmented)
        ref = torch.empty(B, H, S, D, dtype=torch.bfloat16, device=q.device)
        ref_lse = torch.empty(B, H, S, device=q.device) \
            if score == bsm.SCORE_SOFTMAX else None
        bsm.bsm_splash_fwd(q, k, v, info, seg, seg, scale, score, ref, ref_lse)
        torch.cuda.synchronize()
        assert bsm.bsm_device_status()[0] == 0
        for call in range(2):
            out = torch.full_like(ref, float("nan"))
            lse = torch.full_like(ref_lse, float("nan")) \
                if ref_lse is not None else None
            _noalloc(q, k, v, info, seg, scale, score, out, lse)
            torch.cuda.synchronize()
            assert bsm.bsm_device_status()[0] == 0
            what = f"S={S} D={D} call {call}"
            assert torch.equal(out, ref), what
            if lse is not None:
                assert torch.equal(lse, ref_lse), what


def test_noalloc_takes_no_device_memory_after_first_call():
    q, k, v, seg, info = _problem(1, 4, 2048, 128, 61, True)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device)
    # the first call in this context may load the library's device code
    _noalloc(q, k, v, info, seg, 0.1, bsm.SCORE_SOFTMAX, out, lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        _noalloc(q, k, v, info, seg, 0.1, bsm.SCORE_SOFTMAX, out, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1}"
    assert bsm.bsm_device_status()[0] == 0
