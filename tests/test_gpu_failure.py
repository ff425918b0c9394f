"""Failure detection without a GPU fault: a bounded wait that must run out
reports BSM_ERR_DEVICE_TIMEOUT through bsm_device_status, and the context
stays usable afterwards."""

import math

import pytest
import torch

import block_sparse_masked_build_gb300 as bsm
from gpu_helpers import run_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    st, _ = bsm.bsm_device_status()
    assert st == 0
    bsm.bsm_selftest_wait_timeout(2_000_000)  # 2 ms, nothing ever arrives
    st, detail = bsm.bsm_device_status()
    assert st == -4, (st, detail)
    assert detail[0] == 1 and detail[3] == 7
    # the record is cleared by the read
    st, _ = bsm.bsm_device_status()
    assert st == 0


def test_context_usable_after_timeout():
    bsm.bsm_selftest_wait_timeout(1_000_000)
    assert bsm.bsm_device_status()[0] == -4
    g = torch.Generator().manual_seed(1)
    q = torch.randn(1, 1, 256, 128, generator=g).to(torch.bfloat16)
    out, lse, _ = run_gpu(q, q, q, bsm.MASK_CAUSAL, 0, None, None,
                          1 / math.sqrt(128), bsm.SCORE_SOFTMAX)
    assert torch.isfinite(out).all()
    # causal row 0 sees only key 0
    assert torch.equal(out[0, 0, 0].to(torch.bfloat16), q[0, 0, 0])
