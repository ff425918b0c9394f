"""Forward kernel (through the C ABI) vs the fp64 oracle.

Small cases are compared on every output element; they span several
128-row tiles and KV tiles and end in ragged tails.  The full-size workloads
run in the launch configuration the benchmark times and are compared on
every output row (one row per 128-row query tile of every head for the
S=32768 local window).
"""

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import block_sparse_masked_build_gb300 as bsm
from block_sparse_masked_build_gb300 import workloads as wl
from gpu_helpers import compare_lse, compare_out, run_gpu, workload_inputs

pytestmark = pytest.mark.gpu

C, L, SG, BD, DN = (bsm.MASK_CAUSAL, bsm.MASK_LOCAL, bsm.MASK_SEGMENT,
                     bsm.MASK_BAND, bsm.MASK_DENSE)
SM, PW = bsm.SCORE_SOFTMAX, bsm.SCORE_POINTWISE


def _qkv(B, H, Hkv, Sq, Skv, D, seed, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, D, generator=g) * sigma).to(torch.bfloat16)
    k = (torch.randn(B, Hkv, Skv, D, generator=g) * sigma).to(torch.bfloat16)
    v = (torch.randn(B, Hkv, Skv, D, generator=g) * sigma).to(torch.bfloat16)
    return q, k, v


def _expand_kv(t, H):
    g = H // t.shape[1]
    return t.repeat_interleave(g, dim=1)


def _check_full(q, k, v, flags, window, sq, skv, scale, score, **kw):
    out, lse, _ = run_gpu(q, k, v, flags, window, sq, skv, scale, score, **kw)
    H = q.shape[1]
    ke, ve = _expand_kv(k, H), _expand_kv(v, H)
    dense = kw.get("dense")
    if score == SM:
        ref, ref_lse = oracle.softmax_attention(q, ke, ve, flags, window, sq,
                                                skv, scale, dense=dense)
        compare_out(out.numpy(), ref, what="softmax")
        compare_lse(lse.numpy(), ref_lse, what="lse")
    else:
        ref = oracle.pointwise_attention(q, ke, ve, flags, window, sq, skv,
                                         scale, dense=dense)
        compare_out(out.numpy(), ref, pointwise=True, what="pointwise")
    return out, lse


SMALL = [
    # name, B, H, Hkv, Sq, Skv, D, flags, window, score, bq, bkv
    ("cfg1", 1, 2, 2, 256, 256, 64, C, 0, SM, 64, 64),
    ("causal_ragged_pair", 1, 2, 2, 384, 384, 128, C, 0, SM, 128, 128),
    ("causal_tail", 2, 1, 1, 300, 300, 128, C, 0, SM, 128, 128),
    ("full_cross", 1, 2, 2, 200, 333, 128, 0, 0, SM, 128, 128),
    ("full_cross_d64", 2, 1, 1, 130, 520, 64, 0, 0, SM, 64, 128),
    ("local_ragged", 1, 2, 2, 1000, 1000, 128, C | L, 300, SM, 128, 128),
    ("local_bq64", 1, 1, 1, 777, 777, 64, C | L, 129, SM, 64, 64),
    ("symmetric_band", 1, 1, 1, 600, 600, 128, L, 100, SM, 128, 128),
    ("pointwise_causal", 1, 2, 2, 384, 384, 128, C, 0, PW, 128, 128),
    ("pointwise_full_d64", 1, 2, 2, 256, 200, 64, 0, 0, PW, 64, 64),
    ("gqa", 1, 4, 2, 512, 512, 128, C, 0, SM, 128, 128),
    ("blocks_256", 1, 2, 2, 768, 768, 128, C, 0, SM, 256, 256),
    ("blocks_mixed", 1, 2, 2, 640, 640, 128, C, 0, SM, 64, 256),
    # at least 4096 keys without segments: the kernel whose score warps
    # alternate softmax turns between the two query tiles
    ("long_causal_pingpong", 1, 1, 1, 4096, 4096, 128, C, 0, SM, 128, 128),
    ("long_local_pingpong", 1, 1, 1, 4500, 4500, 128, C | L, 1500, SM, 128,
     128),
    ("long_pointwise_pingpong", 1, 1, 1, 4096, 4096, 128, C, 0, PW, 128, 128),
    # symmetric sliding window |q - k| < W
    ("band_softmax", 1, 2, 2, 700, 700, 128, L | BD, 150, SM, 128, 128),
    ("band_ragged_b64", 1, 1, 1, 333, 333, 64, L | BD, 40, SM, 64, 64),
    ("band_pointwise", 1, 2, 2, 640, 640, 128, L | BD, 200, PW, 128, 128),
    ("band_long_pingpong", 1, 1, 1, 4224, 4224, 128, L | BD, 700, SM, 128,
     128),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_cases_elementwise(case):
    name, B, H, Hkv, Sq, Skv, D, flags, window, score, bq, bkv = case
    q, k, v = _qkv(B, H, Hkv, Sq, Skv, D, seed=zlib.crc32(name.encode()) % 10000,
                   sigma=0.5 if score == PW else 1.0)
    _check_full(q, k, v, flags, window, None, None, 1 / math.sqrt(D), score,
                block_q=bq, block_kv=bkv)


@pytest.mark.parametrize("score", [SM, PW])
@pytest.mark.parametrize("extra", [0, C])
def test_dense_mask_elementwise(score, extra):
    # an arbitrary bit-packed mask (empty, full and random 64x64 tiles),
    # alone or with causal, ragged at both ends
    B, H, Sq, Skv, D = 2, 2, 700 if extra else 500, 700 if extra else 650, 128
    q, k, v = _qkv(B, H, H, Sq, Skv, D, seed=22,
                   sigma=0.5 if score == PW else 1.0)
    dm = wl.random_dense_mask(Sq, Skv, 0.3, 64, 23)
    _check_full(q, k, v, DN | extra, 0, None, None, 0.1, score, dense=dm,
                dense_row_words=24)


def test_dense_mask_with_segments_and_long_keys_elementwise():
    # arbitrary mask AND packed segments, and alone at 4224 keys
    B, H, S, D = 1, 1, 4224, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=24)
    dm = wl.random_dense_mask(S, S, 0.5, 128, 25)
    seg = wl.random_segment_ids(B, S, 500, 2000, 26)
    _check_full(q, k, v, DN | SG | C, 0, seg, seg, 0.1, SM, dense=dm)
    _check_full(q, k, v, DN | C, 0, None, None, 0.1, SM, dense=dm)


def test_symmetric_window_with_segments_elementwise():
    B, H, S, D = 2, 2, 900, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=17)
    seg = wl.random_segment_ids(B, S, 50, 400, 18)
    _check_full(q, k, v, L | BD | SG, 120, seg, seg, 0.1, SM)


# head dim 64 under every per-element mask kind, and grouped K/V heads under
# the pointwise path and segment ids ([HSTU] _apply_mask; [NOTES] section 21
# query head h reads K/V head h // (H / H_kv)).
SEG_CASES = [
    # name, B, H, Hkv, S, D, flags, score, seg kind
    ("d64_packed_causal", 2, 2, 2, 700, 64, C | SG, SM, "sorted"),
    ("d64_packed_full", 1, 2, 2, 520, 64, SG, SM, "sorted"),
    ("d64_unsorted", 1, 2, 2, 512, 64, C | SG, SM, "unsorted"),
    ("d64_packed_pointwise", 2, 2, 2, 640, 64, C | SG, PW, "sorted"),
    ("d64_unsorted_pointwise", 1, 2, 2, 384, 64, SG, PW, "unsorted"),
    ("gqa_pointwise", 1, 4, 2, 640, 128, C, PW, None),
    ("gqa_packed", 2, 4, 1, 900, 128, C | SG, SM, "sorted"),
    ("gqa_packed_pointwise", 1, 6, 2, 768, 128, C | SG, PW, "sorted"),
    ("gqa_d64_packed", 1, 4, 2, 600, 64, C | SG, SM, "sorted"),
]


@pytest.mark.parametrize("case", SEG_CASES, ids=[c[0] for c in SEG_CASES])
def test_segment_and_gqa_cases_elementwise(case):
    name, B, H, Hkv, S, D, flags, score, kind = case
    seed = zlib.crc32(name.encode()) % 10000
    q, k, v = _qkv(B, H, Hkv, S, S, D, seed=seed,
                   sigma=0.5 if score == PW else 1.0)
    seg = None
    if kind == "sorted":
        seg = wl.random_segment_ids(B, S, 30, 260, seed + 1)
    elif kind == "unsorted":
        seg = np.random.default_rng(seed + 2).integers(
            0, 3, size=(B, S)).astype(np.int32)
    bq = 64 if D == 64 else 128
    _check_full(q, k, v, flags, 0, seg, seg, 1 / math.sqrt(D), score,
                block_q=bq, block_kv=bq)


@pytest.mark.parametrize("score", [SM, PW])
def test_dense_mask_d64_elementwise(score):
    # an arbitrary mask at head dim 64, alone and with packed segments
    B, H, S, D = 2, 2, 600, 64
    q, k, v = _qkv(B, H, H, S, S, D, seed=27,
                   sigma=0.5 if score == PW else 1.0)
    dm = wl.random_dense_mask(S, S, 0.4, 64, 28)
    _check_full(q, k, v, DN | C, 0, None, None, 0.125, score, dense=dm,
                block_q=64, block_kv=64)
    seg = wl.random_segment_ids(B, S, 40, 300, 29)
    _check_full(q, k, v, DN | SG, 0, seg, seg, 0.125, score, dense=dm,
                block_q=64, block_kv=64)


@pytest.mark.parametrize("score", [SM, PW])
@pytest.mark.parametrize("causal", [True, False])
def test_packed_segments_elementwise(score, causal):
    B, H, S, D = 2, 2, 640, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=5, sigma=0.5 if score == PW else 1)
    seg = wl.random_segment_ids(B, S, 20, 300, 9)
    flags = SG | (C if causal else 0)
    _check_full(q, k, v, flags, 0, seg, seg, 0.09, score)


def test_unsorted_segment_ids_elementwise():
    B, H, S, D = 1, 2, 512, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=6)
    rng = np.random.default_rng(3)
    seg = rng.integers(0, 3, size=(B, S)).astype(np.int32)
    _check_full(q, k, v, C | SG, 0, seg, seg, 0.1, SM)


def test_fully_masked_rows_give_zero_and_neg_inf():
    B, H, S, D = 1, 1, 256, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=7)
    qseg = np.zeros((1, S), dtype=np.int32)
    qseg[0, 30:170] = 9
    kvseg = np.zeros((1, S), dtype=np.int32)
    out, lse = _check_full(q, k, v, SG, 0, qseg, kvseg, 0.1, SM)
    assert torch.all(out[0, 0, 30:170] == 0)
    assert torch.all(torch.isneginf(lse[0, 0, 30:170]))


def test_empty_keys():
    B, H, Sq, D = 1, 2, 200, 128
    q, _, _ = _qkv(B, H, H, Sq, 1, D, seed=8)
    k = torch.empty(B, H, 0, D, dtype=torch.bfloat16)
    out, lse, _ = run_gpu(q, k, k.clone(), 0, 0, None, None, 0.1, SM)
    assert torch.all(out == 0)
    assert torch.all(torch.isneginf(lse))


def test_bshd_layout_matches():
    B, H, S, D = 2, 3, 384, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=9)
    a, la, _ = run_gpu(q, k, v, C, 0, None, None, 0.1, SM)
    b, lb, _ = run_gpu(q, k, v, C, 0, None, None, 0.1, SM, layout="bshd")
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("score", [SM, PW])
def test_block_size_independence(score):
    # the result must not depend on the mask-info block sizes
    B, H, S, D = 1, 2, 512, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=10, sigma=0.5 if score == PW else 1)
    seg = wl.random_segment_ids(B, S, 30, 200, 11)
    outs = []
    for bq, bkv in [(64, 64), (128, 128), (256, 256), (64, 128), (128, 32)]:
        o, l, _ = run_gpu(q, k, v, C | SG, 0, seg, seg, 0.1, score,
                          block_q=bq, block_kv=bkv)
        outs.append((o, l))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0])
        if score == SM:
            assert torch.equal(l, outs[0][1])


@pytest.mark.parametrize("flags", [C | SG, C])
def test_unit_order_does_not_change_results(flags):
    # longest-first and fallback schedules give bit-identical outputs
    B, H, S, D = 2, 3, 1000, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=13)
    seg = wl.random_segment_ids(B, S, 40, 400, 14) if flags & SG else None
    a, la, ia = run_gpu(q, k, v, flags, 0, seg, seg, 0.1, SM)
    assert ia.super_order is not None
    b, lb, _ = run_gpu(q, k, v, flags, 0, seg, seg, 0.1, SM,
                       longest_first=False)
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("D", [64, 128])
def test_padded_output_rows_match(D):
    # an output row stride of D + 8 elements (16-byte but not 32-byte
    # aligned rows) takes the narrower store path; results are identical
    B, H, S = 1, 2, 384
    q, k, v = _qkv(B, H, H, S, S, D, seed=15)
    a, la, info = run_gpu(q, k, v, C, 0, None, None, 0.1, SM)
    dev = torch.device("cuda")
    big = torch.full((B, H, S, D + 8), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    out = big[..., :D]
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    bsm.bsm_splash_fwd(q.to(dev), k.to(dev), v.to(dev), info, None, None, 0.1,
                       SM, out, lse)
    torch.cuda.synchronize()
    assert torch.equal(out.float().cpu(), a) and torch.equal(lse.cpu(), la)
    assert torch.isnan(big[..., D:].float()).all()


def test_repeated_calls_are_deterministic():
    B, H, S, D = 2, 4, 1024, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=12)
    a, la, _ = run_gpu(q, k, v, C, 0, None, None, 0.1, SM)
    b, lb, _ = run_gpu(q, k, v, C, 0, None, None, 0.1, SM)
    assert torch.equal(a, b) and torch.equal(la, lb)


# Full-size workloads in the benchmark's launch configuration, compared with
# the oracle on EVERY output row (about 25 s of host time per S=8192 or
# S=4096 workload), except the S=32768 local window, where one seeded row of
# every 128-row query tile of every (batch, head) is compared, plus the rows
# where the window starts to cut (4095, 4096, 4097) and the first and last.
FULL_ALL_ROWS = ["cfg1_causal_s256_d64", "cfg2_causal_s2048_d128",
                 "cfg3_packed_s8192_d128", "cfg3c_causal_s8192_d128",
                 "cfg4_hstu_s4096_d128", "cfg4p_hstu_s4096_d128",
                 "next3_band_s8192_d128", "next2_dense_s8192_d128"]


def _full_size_run(name):
    w, q, k, v, seg = workload_inputs(name)
    dm = wl.make_dense_mask(w)
    out, lse, _ = run_gpu(q, k, v, w.flags, w.window, seg, seg, w.scale,
                          w.score, block_q=w.block_q, block_kv=w.block_kv,
                          dense=dm)
    return w, q, k, v, seg, dm, out, lse


def _full_size_properties(w, dm, out, lse):
    # at any size: outputs are finite, and lse is finite exactly on the rows
    # that see at least one key (a row an arbitrary mask hides completely
    # gives out = 0 and lse = -inf)
    assert torch.isfinite(out).all()
    if w.score != SM:
        return
    if dm is None:
        assert torch.isfinite(lse).all()
        return
    from block_sparse_masked_build_gb300 import flops as fl
    seen = fl.visible_pairs_per_row(w.flags, w.window, w.Sq, w.Skv_,
                                    dense=dm) > 0
    seen = torch.from_numpy(seen)
    assert torch.isfinite(lse[:, :, seen]).all()
    assert (lse[:, :, ~seen] == float("-inf")).all()
    assert (out[:, :, ~seen] == 0).all()


@pytest.mark.parametrize("name", FULL_ALL_ROWS)
def test_full_size_workloads_every_row(name):
    w, q, k, v, seg, dm, out, lse = _full_size_run(name)
    _full_size_properties(w, dm, out, lse)
    if w.score == SM:
        ref, ref_lse = oracle.softmax_attention(q, k, v, w.flags, w.window,
                                                seg, seg, w.scale, dense=dm)
        compare_out(out.numpy(), ref, what=name)
        compare_lse(lse.numpy(), ref_lse, what=name)
    else:
        ref = oracle.pointwise_attention(q, k, v, w.flags, w.window, seg, seg,
                                         w.scale, dense=dm)
        compare_out(out.numpy(), ref, pointwise=True, what=name)


def test_full_size_local_window_every_tile():
    name = "cfg5_local_s32768_d128"
    w, q, k, v, seg, dm, out, lse = _full_size_run(name)
    _full_size_properties(w, dm, out, lse)
    rng = np.random.default_rng(321)
    rows = set()
    for b in range(w.B):
        for h in range(w.H):
            for t0 in range(0, w.Sq, 128):
                rows.add((b, h, t0 + int(rng.integers(min(128, w.Sq - t0)))))
            for r in (0, w.window - 1, w.window, w.window + 1, w.Sq - 1):
                rows.add((b, h, r))
    rows = sorted(rows)
    got = np.stack([out[b, h, r].numpy() for (b, h, r) in rows])
    ref, ref_lse = oracle.softmax_attention(q, k, v, w.flags, w.window, seg,
                                            seg, w.scale, rows=rows)
    compare_out(got, ref, what=name)
    compare_lse(np.array([lse[b, h, r].item() for (b, h, r) in rows]),
                ref_lse, what=name)


def test_constant_value_rows_full_size():
    # invariant at full size (packed segments): constant v rows -> that row
    w, q, k, _, seg = workload_inputs("cfg3_packed_s8192_d128")
    c = torch.linspace(-1.5, 2.0, w.D).to(torch.bfloat16)
    v = c.expand(w.B, w.H, w.S, w.D).contiguous()
    out, _, _ = run_gpu(q, k, v, w.flags, 0, seg, seg, w.scale, SM)
    err = (out - c.float()).abs().max().item()
    assert err <= 2e-2


@pytest.mark.parametrize("score", [SM, PW])
def test_many_repeats_bitwise_identical(score):
    # The P.V product of a tile and the next Q.K^T into the same TMEM
    # columns are issued back to back; a reordering would show up as
    # run-to-run differences.  30 launches with thousands of such pairs each.
    B, H, S, D = 1, 8, 4096, 128
    q, k, v = _qkv(B, H, H, S, S, D, seed=13, sigma=0.5 if score == PW else 1)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    info = bsm.build_mask_info(C, B, S, S, 128, 128, device=dev)
    ref = None
    for it in range(30):
        out = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev) \
            if score == SM else None
        bsm.bsm_splash_fwd(qd, kd, vd, info, None, None, 0.09, score, out, lse)
        if ref is None:
            ref = (out.clone(), None if lse is None else lse.clone())
        else:
            assert torch.equal(out, ref[0]), f"run {it} differs"
            if lse is not None:
                assert torch.equal(lse, ref[1]), f"run {it} lse differs"
    torch.cuda.synchronize()
    assert bsm.bsm_device_status()[0] == 0
    rows = [(0, h, r) for h in range(H) for r in (0, 1, 127, 128, 2047, 4095)]
    got = np.stack([ref[0][b, h, r].float().cpu().numpy() for b, h, r in rows])
    if score == SM:
        want, _ = oracle.softmax_attention(q, k, v, C, 0, None, None, 0.09,
                                           rows=rows)
        compare_out(got, want, what="repeat")
    else:
        want = oracle.pointwise_attention(q, k, v, C, 0, None, None, 0.09,
                                          rows=rows)
        compare_out(got, want, pointwise=True, what="repeat")


def test_full_size_grouped_heads_every_row_of_sampled_heads():
    # 32 query heads over 8 K/V heads: units pair two heads of a group on
    # the same rows.  Every row of heads from both members of a pair and
    # of different groups and batch rows, against the oracle with the
    # matching K/V head ([NOTES] section 21: head h reads K/V head h // 4).
    name = "next1_gqa_s8192_d128"
    w, q, k, v, seg = workload_inputs(name)
    out, lse, _ = run_gpu(q, k, v, w.flags, w.window, seg, seg, w.scale,
                          w.score)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    G = w.H // w.Hkv_
    for (b, h) in [(0, 0), (0, 1), (0, 6), (1, 19), (1, 31)]:
        kh = slice(h // G, h // G + 1)
        ref, ref_lse = oracle.softmax_attention(
            q[b:b + 1, h:h + 1], k[b:b + 1, kh], v[b:b + 1, kh], w.flags,
            w.window, None, None, w.scale)
        compare_out(out[b:b + 1, h:h + 1].numpy(), ref, what=f"b{b} h{h}")
        compare_lse(lse[b:b + 1, h:h + 1].numpy(), ref_lse, what=f"b{b} h{h}")


def test_maximum_sequence_length_local_window():
    """Sq = Skv = 262144, the longest sequence the kernels take (2048 x 2048
    mask blocks: the mask-info build takes its three-launch path), under a
    local window of 1024 keys, two heads; one row of every 256-row work
    unit is compared with the oracle, at a varying offset in the unit."""
    B, H, S, D = 1, 2, 262144, 64
    q, k, v = _qkv(B, H, H, S, S, D, 4242)
    scale = 1.0 / math.sqrt(D)
    out, lse, _ = run_gpu(q, k, v, L, 1024, None, None, scale, SM)
    units = S // 256
    rows = [(0, u % H, u * 256 + (u * 37) % 256) for u in range(units)]
    ref, ref_lse = oracle.softmax_attention(q, k, v, L, 1024, None, None,
                                            scale, rows=rows)
    got = np.stack([out[b, h, r].float().numpy() for b, h, r in rows])
    got_lse = np.array([lse[b, h, r].item() for b, h, r in rows])
    compare_out(got, ref, what="max-length out")
    compare_lse(got_lse, ref_lse, what="max-length lse")


@pytest.mark.parametrize("n_chunks", [1, 3, 16])
def test_host_entry_chunks_match_device_path(n_chunks):
    """bsm_splash_fwd_host over ragged head ranges (5 K/V heads in 1, 3 or
    5 ranges; grouped query heads, packed segments, a ragged sequence
    length) returns exactly the device path's out and lse, also when two
    calls run back to back on one device buffer with other inputs."""
    B, H, Hkv, S, D = 2, 10, 5, 1000, 128
    flags = C | SG
    dev = torch.device("cuda")
    outs = []
    nbytes = bsm.bsm_splash_fwd_host_bytes(flags, 0, B, H, Hkv, S, S, D, 128,
                                           128, SM)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    cases = []
    for seed in (707, 708):
        q, k, v = (t.pin_memory() for t in _qkv(B, H, Hkv, S, S, D, seed))
        seg = torch.from_numpy(wl.random_segment_ids(B, S, 30, 400, seed))
        seg = seg.pin_memory()
        out = torch.empty((B, H, S, D), dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
        cases.append((q, k, v, seg, out, lse))
    stream = torch.cuda.current_stream()
    for q, k, v, seg, out, lse in cases:   # both enqueued before a sync
        bsm.bsm_splash_fwd_host(flags, 0, q, k, v, seg, seg, 128, 128,
                                1.0 / math.sqrt(D), SM, out, lse, buf,
                                n_chunks, stream)
    stream.synchronize()
    assert bsm.bsm_device_status()[0] == 0
    for q, k, v, seg, out, lse in cases:
        segd = seg.to(dev)
        ref_out, ref_lse = bsm.splash_attention(
            q.to(dev), k.to(dev), v.to(dev), mask_flags=flags,
            q_segment_ids=segd, kv_segment_ids=segd)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out.cpu())
        assert torch.equal(lse, ref_lse.cpu())


@pytest.mark.parametrize("case", ["causal", "segments", "gqa", "pointwise"])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_inputs_match_device_path(case, pinned):
    """splash_attention with host tensors (bsm_splash_fwd_host: copies in
    chunks of heads that overlap the forward when the memory is pinned)
    returns exactly what the same call on device tensors returns."""
    B, H, Hkv, S, D = 2, 8, 8, 1024, 128
    flags, score, seg = C, SM, None
    if case == "segments":
        flags = C | SG
        seg = torch.from_numpy(wl.random_segment_ids(B, S, 40, 500, 5))
    if case == "gqa":
        Hkv = 2
    if case == "pointwise":
        score = PW
    q, k, v = _qkv(B, H, Hkv, S, S, D, 606)
    dev = torch.device("cuda")
    segd = None if seg is None else seg.to(dev)
    ref_out, ref_lse = bsm.splash_attention(
        q.to(dev), k.to(dev), v.to(dev), mask_flags=flags,
        q_segment_ids=segd, kv_segment_ids=segd, score=score)
    torch.cuda.synchronize()
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
        seg = None if seg is None else seg.pin_memory()
    out, lse = bsm.splash_attention(q, k, v, mask_flags=flags,
                                    q_segment_ids=seg, kv_segment_ids=seg,
                                    score=score)
    assert out.device.type == "cpu"
    assert torch.equal(out, ref_out.cpu())
    if score == SM:
        assert torch.equal(lse, ref_lse.cpu())
    else:
        assert lse is None and ref_lse is None
    assert bsm.bsm_device_status()[0] == 0
