"""State the build and the forward keep in caller buffers, and replays.

The one-launch mask-info build counts its CTAs in a word of the caller's
mask-info buffer, which the caller does not initialise: the word carries a
per-build tag, a word with another tag counts as zero, and the last CTA puts
the count back to zero.  The persistent forward takes work units from a
counter in the caller's workspace, zeroed on the stream before its launch.
These tests fill both buffers with leftover bytes before a call, and replay a
CUDA graph of build + forward (the tag is then the same on every replay, so
each launch must leave its count at zero for the next), changing the segment
ids and the queries between replays so that a stale table or a skipped unit
would show.  Outputs are compared with the oracle, and replays bit for bit
with eager calls.
"""

import numpy as np
import pytest
import torch

import oracle
import block_sparse_masked_build_gb300 as bsm
from block_sparse_masked_build_gb300 import workloads as wl
from gpu_helpers import compare_lse, compare_out

pytestmark = pytest.mark.gpu

B, H, S, D = 2, 2, 1536, 128
FLAGS = bsm.MASK_CAUSAL | bsm.MASK_SEGMENT
SCALE = 1.0 / np.sqrt(D)


def _inputs(seed):
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(B, H, S, D, generator=g).to(torch.bfloat16)
               for _ in range(3))
    seg = wl.random_segment_ids(B, S, 60, 900, seed + 1)
    return q, k, v, seg


def _buffers(dev):
    nbytes = bsm.bsm_mask_info_bytes(FLAGS, 0, B, S, S, 128, 128)
    mib = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ws = torch.empty(bsm.bsm_splash_fwd_workspace_bytes(), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    return mib, ws, out, lse


def _step(qd, kd, vd, segd, mib, ws, out, lse):
    info = bsm.bsm_build_mask_info(FLAGS, 0, segd, segd, B, S, S, 128, 128,
                                   mib)
    bsm.bsm_splash_fwd(qd, kd, vd, info, segd, segd, SCALE,
                       bsm.SCORE_SOFTMAX, out, lse, workspace=ws)


def _oracle_check(q, k, v, seg, out, lse):
    ref, ref_lse = oracle.softmax_attention(q, k, v, FLAGS, 0, seg, seg,
                                            SCALE)
    compare_out(out.float().cpu().numpy(), ref, what="out")
    compare_lse(lse.cpu().numpy(), ref_lse, what="lse")


@pytest.mark.parametrize("fill", [0x00, 0xFF, "random"])
def test_leftover_buffer_contents(fill):
    dev = torch.device("cuda")
    q, k, v, seg = _inputs(31)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    segd = torch.from_numpy(seg).to(dev)
    mib, ws, out, lse = _buffers(dev)
    ref_out = ref_lse = None
    for it in range(3):
        for buf in (mib, ws):
            if fill == "random":
                g = torch.Generator(device=dev).manual_seed(7 + it)
                buf.copy_(torch.randint(0, 256, buf.shape, generator=g,
                                        device=dev, dtype=torch.int32)
                          .to(torch.uint8))
            else:
                buf.fill_(fill)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        _step(qd, kd, vd, segd, mib, ws, out, lse)
        torch.cuda.synchronize()
        assert bsm.bsm_device_status()[0] == 0
        if ref_out is None:
            _oracle_check(q, k, v, seg, out, lse)
            ref_out, ref_lse = out.clone(), lse.clone()
        else:
            assert torch.equal(out, ref_out)
            assert torch.equal(lse, ref_lse)


def test_graph_replay_rebuilds_and_recomputes():
    dev = torch.device("cuda")
    cases = [_inputs(41), _inputs(42)]
    qd = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev)
    kd, vd = torch.empty_like(qd), torch.empty_like(qd)
    segd = torch.empty((B, S), dtype=torch.int32, device=dev)
    mib, ws, out, lse = _buffers(dev)

    def load(c):
        q, k, v, seg = c
        qd.copy_(q)
        kd.copy_(k)
        vd.copy_(v)
        segd.copy_(torch.from_numpy(seg))

    # eager results of both cases (the first is also checked with the oracle)
    eager = []
    for n, c in enumerate(cases):
        load(c)
        _step(qd, kd, vd, segd, mib, ws, out, lse)
        torch.cuda.synchronize()
        assert bsm.bsm_device_status()[0] == 0
        if n == 0:
            _oracle_check(*c, out, lse)
        eager.append((out.clone(), lse.clone()))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capturing stream
        load(cases[0])
        _step(qd, kd, vd, segd, mib, ws, out, lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        _step(qd, kd, vd, segd, mib, ws, out, lse)
    torch.cuda.synchronize()

    for n in (0, 1, 1, 0, 1):
        load(cases[n])
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert bsm.bsm_device_status()[0] == 0
        assert torch.equal(out, eager[n][0]), f"replay of case {n}: out"
        assert torch.equal(lse, eager[n][1]), f"replay of case {n}: lse"
