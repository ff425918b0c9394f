"""Backward kernels (through the C ABI) vs the fp64 backward oracle.

Every gradient element is compared, relative to the reference magnitude
(gates in gpu_helpers, derived in test_bwd_rounding).  The forward's own
outputs (out, lse) feed the backward, as they would in training.  Grouped
K/V heads are checked against the oracle on K/V expanded to every query
head, with each K/V head's gradient summed over its group.
"""

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import block_sparse_masked_build_gb300 as bsm
from block_sparse_masked_build_gb300 import workloads as wl
from gpu_helpers import compare_grad, dense_device_bits

pytestmark = pytest.mark.gpu

C, L, SG, BD, DN = (bsm.MASK_CAUSAL, bsm.MASK_LOCAL, bsm.MASK_SEGMENT,
                     bsm.MASK_BAND, bsm.MASK_DENSE)
SM, PW = bsm.SCORE_SOFTMAX, bsm.SCORE_POINTWISE


def _inputs(B, H, Hkv, Sq, Skv, D, seed, sigma):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, D, generator=g) * sigma).to(torch.bfloat16)
    k = (torch.randn(B, Hkv, Skv, D, generator=g) * sigma).to(torch.bfloat16)
    v = (torch.randn(B, Hkv, Skv, D, generator=g) * sigma).to(torch.bfloat16)
    do = torch.randn(B, H, Sq, D, generator=g).to(torch.bfloat16)
    return q, k, v, do


def _gpu_grads(q, k, v, do, flags, window, seg_q, seg_kv, scale, score,
               bq=128, bkv=128, dense=None):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    sq = None if seg_q is None else torch.from_numpy(seg_q).to(dev)
    sk = None if seg_kv is None else torch.from_numpy(seg_kv).to(dev)
    B, H, Sq, D = q.shape
    db = None if dense is None else dense_device_bits(dense)
    info = bsm.build_mask_info(flags, B, Sq, k.shape[2], bq, bkv, window, sq,
                               sk, device=dev, dense_bits=db)
    out, lse = bsm.splash_attention(qd, kd, vd, mask_flags=flags,
                                    window=window, q_segment_ids=sq,
                                    kv_segment_ids=sk, scale=scale,
                                    score=score, mask_info=info)
    dq, dk, dv = bsm.splash_attention_bwd(qd, kd, vd, out, lse, dod,
                                          q_segment_ids=sq, kv_segment_ids=sk,
                                          scale=scale, score=score,
                                          mask_info=info)
    torch.cuda.synchronize()
    st, detail = bsm.bsm_device_status()
    assert st == 0, f"device status {st} {detail}"
    return dq.float().cpu(), dk.float().cpu(), dv.float().cpu()


def _oracle_grads(q, k, v, do, flags, window, seg_q, seg_kv, scale, score,
                  dense=None):
    H, Hkv = q.shape[1], k.shape[1]
    grp = H // Hkv
    ke, ve = k.repeat_interleave(grp, dim=1), v.repeat_interleave(grp, dim=1)
    fn = oracle.softmax_attention_bwd if score == SM else \
        oracle.pointwise_attention_bwd
    dq, dk, dv = fn(q, ke, ve, do, flags, window, seg_q, seg_kv, scale,
                    dense=dense)
    B, _, Skv, D = k.shape
    dk = dk.reshape(B, Hkv, grp, Skv, D).sum(axis=2)
    dv = dv.reshape(B, Hkv, grp, Skv, D).sum(axis=2)
    return dq, dk, dv


def _check(q, k, v, do, flags, window, seg_q, seg_kv, scale, score, **kw):
    got = _gpu_grads(q, k, v, do, flags, window, seg_q, seg_kv, scale, score,
                     **kw)
    ref = _oracle_grads(q, k, v, do, flags, window, seg_q, seg_kv, scale,
                        score, dense=kw.get("dense"))
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        compare_grad(g.numpy(), r, what=name)
    return got


CASES = [
    # name, B, H, Hkv, Sq, Skv, D, flags, window, score, block
    ("causal_ragged", 1, 2, 2, 384, 384, 128, C, 0, SM, 128),
    ("causal_tail_d64", 2, 1, 1, 300, 300, 64, C, 0, SM, 64),
    ("full_cross", 1, 2, 2, 200, 333, 128, 0, 0, SM, 128),
    ("local", 1, 2, 2, 700, 700, 128, C | L, 200, SM, 128),
    ("band", 1, 1, 1, 600, 600, 128, L | BD, 100, SM, 128),
    ("gqa", 1, 4, 2, 512, 512, 128, C, 0, SM, 128),
    ("pointwise_causal", 1, 2, 2, 384, 384, 128, C, 0, PW, 128),
    ("pointwise_full_d64", 1, 2, 2, 256, 200, 64, 0, 0, PW, 64),
    ("pointwise_gqa", 1, 6, 2, 320, 320, 128, C, 0, PW, 128),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_small_cases(case):
    name, B, H, Hkv, Sq, Skv, D, flags, window, score, blk = case
    q, k, v, do = _inputs(B, H, Hkv, Sq, Skv, D,
                          zlib.crc32(name.encode()) % 10000,
                          0.5 if score == PW else 1.0)
    _check(q, k, v, do, flags, window, None, None, 1 / math.sqrt(D), score,
           bq=blk, bkv=blk)


@pytest.mark.parametrize("score", [SM, PW])
@pytest.mark.parametrize("kind", ["sorted", "unsorted"])
@pytest.mark.parametrize("D", [64, 128])
def test_backward_segments(score, kind, D):
    B, H, S = 2, 2, 520
    q, k, v, do = _inputs(B, H, H, S, S, D, 40 + D + score,
                          0.5 if score == PW else 1.0)
    if kind == "sorted":
        seg = wl.random_segment_ids(B, S, 30, 250, 41)
    else:
        seg = np.random.default_rng(42).integers(0, 3, size=(B, S)).astype(
            np.int32)
    _check(q, k, v, do, C | SG, 0, seg, seg, 0.1, score, bq=64, bkv=64)


@pytest.mark.parametrize("score", [SM, PW])
def test_backward_arbitrary_mask(score):
    B, H, S, D = 1, 2, 500, 128
    q, k, v, do = _inputs(B, H, H, S, S, D, 50 + score,
                          0.5 if score == PW else 1.0)
    dm = wl.random_dense_mask(S, S, 0.4, 64, 51)
    _check(q, k, v, do, DN | C, 0, None, None, 0.1, score, dense=dm)


def test_backward_rows_that_see_nothing():
    # query rows whose segment id no key has: zero dq; keys no query sees:
    # zero dk and dv
    B, H, S, D = 1, 1, 256, 128
    q, k, v, do = _inputs(B, H, H, S, S, D, 60, 1.0)
    qseg = np.zeros((1, S), dtype=np.int32)
    qseg[0, 30:170] = 9
    kvseg = np.zeros((1, S), dtype=np.int32)
    kvseg[0, 200:] = 7
    dq, dk, dv = _check(q, k, v, do, SG, 0, qseg, kvseg, 0.1, SM)
    assert torch.all(dq[0, 0, 30:170] == 0)
    assert torch.all(dk[0, 0, 200:] == 0) and torch.all(dv[0, 0, 200:] == 0)


def test_backward_block_size_independence():
    B, H, S, D = 1, 2, 512, 128
    q, k, v, do = _inputs(B, H, H, S, S, D, 70, 1.0)
    seg = wl.random_segment_ids(B, S, 30, 200, 71)
    outs = [_gpu_grads(q, k, v, do, C | SG, 0, seg, seg, 0.1, SM, bq=bq,
                       bkv=bkv)
            for bq, bkv in [(64, 64), (128, 128), (256, 128)]]
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["cfg2_causal_s2048_d128",
                                  "cfg3_packed_s8192_d128",
                                  "cfg4p_hstu_s4096_d128"])
def test_backward_full_size_sampled_heads(name):
    # full-size workload through the GPU; the oracle on three (batch, head)
    # pairs (every element of their gradients)
    w = wl.WORKLOADS[name]
    q, k, v = wl.make_qkv(w)
    g = torch.Generator().manual_seed(w.seed + 7)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    seg = wl.make_segment_ids(w)
    got = _gpu_grads(q, k, v, do, w.flags, w.window, seg, seg, w.scale,
                     w.score, bq=w.block_q, bkv=w.block_kv)
    for (b, h) in [(0, 0), (w.B - 1, w.H // 2), (w.B // 2, w.H - 1)]:
        sl = slice(b, b + 1), slice(h, h + 1)
        sb = None if seg is None else seg[b:b + 1]
        ref = _oracle_grads(q[sl], k[sl], v[sl], do[sl], w.flags, w.window,
                            sb, sb, w.scale, w.score)
        for nm, gv, r in zip(("dq", "dk", "dv"), got, ref):
            compare_grad(gv[sl].numpy(), r, what=f"{name} {nm} b{b} h{h}")
