"""Pins of the oracle's mask-info (block classes, next-block table, lists).

The oracle classifies blocks by scanning every element.  These tests derive
the same classes a different way -- from the range of q - k over a block
(causal / local masks) or from segment intervals (packed sequences) -- and
check closed-form counts and the worked example of the splash notes
(section 21).
"""

import os

import numpy as np
import pytest

import oracle
from oracle import MASK_BAND, MASK_CAUSAL, MASK_LOCAL, MASK_SEGMENT
from block_sparse_masked_build_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _interval_classes(flags, window, Sq, Skv, bq, bkv):
    """Classes of causal/local masks from the q-k range of each block.

    Rows r0..r1 and columns c0..c1 (clipped to the sequence) give every
    integer d = q - k in [r0 - c1, r1 - c0].  Causal needs d >= 0, local
    d < W.  The block is nonempty iff that range meets the allowed one, full
    iff it lies inside it and the block is not cut by the sequence end.
    """
    nq, nk = -(-Sq // bq), -(-Skv // bkv)
    lo_ok = 0 if flags & MASK_CAUSAL else (
        1 - window if flags & MASK_BAND else -10**9)
    hi_ok = (window - 1) if flags & MASK_LOCAL else 10**9
    cls = np.zeros((nq, nk), dtype=np.int8)
    for i in range(nq):
        r0, r1 = i * bq, min(Sq, (i + 1) * bq) - 1
        for j in range(nk):
            c0, c1 = j * bkv, min(Skv, (j + 1) * bkv) - 1
            dmin, dmax = r0 - c1, r1 - c0
            if dmax < lo_ok or dmin > hi_ok:
                continue
            ragged = (r1 - r0 + 1 != bq) or (c1 - c0 + 1 != bkv)
            full = dmin >= lo_ok and dmax <= hi_ok and not ragged
            cls[i, j] = 2 if full else 1
    return cls


@pytest.mark.parametrize("Sq,Skv,bq,bkv", [
    (256, 256, 64, 64), (512, 512, 128, 128), (512, 512, 64, 128),
    (512, 512, 128, 64), (300, 300, 64, 64), (384, 520, 128, 128),
    (1000, 1000, 128, 64), (64, 64, 64, 64), (16, 48, 16, 16)])
@pytest.mark.parametrize("flags,window", [
    (MASK_CAUSAL, 0), (MASK_CAUSAL | MASK_LOCAL, 200),
    (MASK_CAUSAL | MASK_LOCAL, 64), (MASK_CAUSAL | MASK_LOCAL, 1), (0, 0),
    (MASK_LOCAL, 150), (MASK_LOCAL | MASK_BAND, 150),
    (MASK_LOCAL | MASK_BAND, 1), (MASK_LOCAL | MASK_BAND, 64)])
def test_classes_match_interval_derivation(Sq, Skv, bq, bkv, flags, window):
    mi = oracle.mask_info(flags, window, None, None, 1, Sq, Skv, bq, bkv)
    ref = _interval_classes(flags, window, Sq, Skv, bq, bkv)
    np.testing.assert_array_equal(mi["block_mask"][0], ref)


def _segment_classes(lens, causal, bq, bkv):
    """Classes of a (causal AND) same-segment mask from segment intervals."""
    S = sum(lens)
    starts = np.cumsum([0] + lens[:-1])
    nq, nk = -(-S // bq), -(-S // bkv)
    cls = np.zeros((nq, nk), dtype=np.int8)
    for i in range(nq):
        r0, r1 = i * bq, min(S, (i + 1) * bq) - 1
        for j in range(nk):
            c0, c1 = j * bkv, min(S, (j + 1) * bkv) - 1
            nonempty = False
            for a, n in zip(starts, lens):
                b = a + n - 1
                qlo, qhi = max(a, r0), min(b, r1)
                klo, khi = max(a, c0), min(b, c1)
                if qlo > qhi or klo > khi:
                    continue
                if not causal or klo <= qhi:
                    nonempty = True
                    break
            if not nonempty:
                continue
            # full: one segment covers all rows and columns (and causal holds
            # for the top-right corner), and the block is not ragged
            one = any(a <= min(r0, c0) and a + n - 1 >= max(r1, c1)
                      for a, n in zip(starts, lens))
            ragged = (r1 - r0 + 1 != bq) or (c1 - c0 + 1 != bkv)
            full = one and not ragged and (not causal or c1 <= r0)
            cls[i, j] = 2 if full else 1
    return cls


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("bq,bkv", [(64, 64), (128, 128), (64, 128)])
def test_segment_classes_match_interval_derivation(seed, causal, bq, bkv):
    rng = np.random.default_rng(seed)
    S = 1024 + 64 * seed + (37 if seed == 2 else 0)
    lens = wl.segment_lengths(rng, S, 20, 300)
    seg = np.repeat(np.arange(len(lens), dtype=np.int32), lens)[None]
    flags = MASK_SEGMENT | (MASK_CAUSAL if causal else 0)
    mi = oracle.mask_info(flags, 0, seg, seg, 1, S, S, bq, bkv)
    np.testing.assert_array_equal(mi["block_mask"][0],
                                  _segment_classes(lens, causal, bq, bkv))


def test_causal_closed_form_counts():
    # square blocks: nq(nq+1)/2 nonzero blocks, nq of them partial (diagonal)
    for S, b in [(2048, 128), (8192, 128), (256, 64), (4096, 128)]:
        mi = oracle.mask_info(MASK_CAUSAL, 0, None, None, 1, S, S, b, b)
        nq = S // b
        bm = mi["block_mask"]
        assert int((bm > 0).sum()) == nq * (nq + 1) // 2
        assert int((bm == 1).sum()) == nq
        assert len(mi["kv_idx"]) == nq * (nq + 1) // 2


def test_local_window_counts_closed_form():
    # S=32768, 128x128 blocks, causal AND q-k < 4096 (32 blocks):
    # row i >= 32 has blocks i-32..i (33 nonzero, the two ends partial);
    # row i < 32 has blocks 0..i (i+1 nonzero, only the diagonal partial).
    S, b, W = 32768, 128, 4096
    nq, w = S // b, W // b
    nonzero = sum(i + 1 for i in range(w)) + (nq - w) * (w + 1)
    partial = w + (nq - w) * 2
    assert (nonzero, partial) == (7920, 480)
    mi = oracle.mask_info(MASK_CAUSAL | MASK_LOCAL, W, None, None, 1, S, S, b,
                          b)
    bm = mi["block_mask"]
    assert int((bm > 0).sum()) == nonzero
    assert int((bm == 1).sum()) == partial
    assert bm.size == 65536


def test_visible_pair_closed_forms():
    S = 2048
    assert oracle.visible_pair_count(MASK_CAUSAL, 0, None, None, 1, S, S) \
        == S * (S + 1) // 2
    # local window: (S - W) rows see W keys, the first W rows see q+1 keys
    S, W = 8192, 1024
    assert oracle.visible_pair_count(MASK_CAUSAL | MASK_LOCAL, W, None, None,
                                     1, S, S) == (S - W) * W + W * (W + 1) // 2
    # the long local-window workload's per-head count
    S, W = 32768, 4096
    assert (S - W) * W + W * (W + 1) // 2 == 125_831_168
    # packed segments: sum of n(n+1)/2 over segments
    lens = [300, 1000, 17, 555]
    seg = np.repeat(np.arange(4, dtype=np.int32), lens)[None]
    assert oracle.visible_pair_count(MASK_CAUSAL | MASK_SEGMENT, 0, seg, seg,
                                     1, sum(lens), sum(lens)) == \
        sum(n * (n + 1) // 2 for n in lens)


def test_band_window_closed_forms():
    # |q - k| < W: row q sees min(q, W-1) + min(S-1-q, W-1) + 1 keys
    for S, W in [(1000, 1), (1000, 37), (4096, 512), (300, 5000)]:
        want = sum(min(q, W - 1) + min(S - 1 - q, W - 1) + 1
                   for q in range(S))
        assert oracle.visible_pair_count(MASK_LOCAL | MASK_BAND, W, None,
                                         None, 1, S, S) == want
    # square blocks of size b with W = b: row i has blocks i-1, i, i+1; the
    # diagonal block is full (|q - k| <= b-1 < W there), its neighbours
    # partial (each holds the pair |q - k| = b)
    S, b = 1024, 128
    nq = S // b
    mi = oracle.mask_info(MASK_LOCAL | MASK_BAND, b, None, None, 1, S, S, b, b)
    bm = mi["block_mask"][0]
    assert int((bm > 0).sum()) == 3 * nq - 2
    assert int((bm == 2).sum()) == nq
    np.testing.assert_array_equal(np.diag(bm), np.full(nq, 2))
    # the band is symmetric; with causal it adds nothing
    vis = oracle.visibility_matrix(MASK_LOCAL | MASK_BAND, 9, 60, 60)
    np.testing.assert_array_equal(vis, vis.T)
    a = oracle.visibility_matrix(MASK_CAUSAL | MASK_LOCAL | MASK_BAND, 9, 60,
                                 60)
    np.testing.assert_array_equal(
        a, oracle.visibility_matrix(MASK_CAUSAL | MASK_LOCAL, 9, 60, 60))


@pytest.mark.parametrize("Sq,Skv,bq,bkv,seed", [
    (256, 256, 64, 64, 1), (300, 200, 32, 64, 2), (128, 520, 128, 128, 3),
    (97, 97, 16, 32, 4)])
def test_dense_mask_classes_from_block_counts(Sq, Skv, bq, bkv, seed):
    # classes straight from the mask: pad it to whole blocks with False,
    # count the set elements of each block by reshaping
    dm = wl.random_dense_mask(Sq, Skv, 0.4, 32, seed)
    nq, nk = -(-Sq // bq), -(-Skv // bkv)
    pad = np.zeros((nq * bq, nk * bkv), dtype=bool)
    pad[:Sq, :Skv] = dm
    cnt = pad.reshape(nq, bq, nk, bkv).sum(axis=(1, 3))
    want = np.where(cnt == 0, 0, np.where(cnt == bq * bkv, 2, 1))
    mi = oracle.mask_info(oracle.MASK_DENSE, 0, None, None, 1, Sq, Skv, bq,
                          bkv, dense=dm)
    np.testing.assert_array_equal(mi["block_mask"][0], want)


def test_dense_pack_round_trip():
    dm = wl.random_dense_mask(70, 100, 0.5, 16, 9)
    words = wl.pack_dense_mask(dm, row_words=5)
    assert words.shape == (70, 5) and words.dtype == np.uint32
    k = np.arange(100)
    back = ((words[:, k // 32] >> (k % 32).astype(np.uint32)) & 1).astype(bool)
    np.testing.assert_array_equal(back, dm)
    assert not words[:, 4].any() and not (words[:, 3] >> 4).any()


def test_closed_form_flop_counts_match_oracle_counts():
    # flops.py's per-row counting (used by the benchmark) against the
    # oracle's element scan, for the band and arbitrary masks
    from block_sparse_masked_build_gb300 import flops as fl
    for flags, W in [(MASK_LOCAL | MASK_BAND, 37),
                     (MASK_LOCAL | MASK_BAND | MASK_CAUSAL, 50)]:
        assert fl.visible_pairs(flags, W, 1, 300, 300) == \
            oracle.visible_pair_count(flags, W, None, None, 1, 300, 300)
    dm = wl.random_dense_mask(300, 260, 0.4, 32, 3)
    for flags in (oracle.MASK_DENSE, oracle.MASK_DENSE | MASK_CAUSAL):
        assert fl.visible_pairs(flags, 0, 1, 300, 260, dense=dm) == \
            oracle.visible_pair_count(flags, 0, None, None, 1, 300, 260,
                                      dense=dm)
    seg = wl.random_segment_ids(2, 300, 20, 90, 4)
    dm = wl.random_dense_mask(300, 300, 0.5, 32, 5)
    flags = oracle.MASK_DENSE | MASK_SEGMENT | MASK_CAUSAL
    assert fl.visible_pairs(flags, 0, 2, 300, 300, seg, seg, dense=dm) == \
        oracle.visible_pair_count(flags, 0, seg, seg, 2, 300, 300, dense=dm)


def _read_golden():
    valid, printed = None, []
    with open(os.path.join(GOLDEN, "data_next_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            nums = [int(x) for x in val.split()]
            if key == "valid":
                valid = nums
            elif key == "printed":
                printed.append(tuple(nums))
    return valid, printed


def test_data_next_worked_example():
    valid, printed = _read_golden()
    bkv = 16
    nk = len(valid)
    # one q block of 16 rows, all in segment 7; kv block j is in segment 7
    # iff it is valid
    q_seg = np.full((1, 16), 7, dtype=np.int32)
    kv_seg = np.repeat(np.where(np.asarray(valid) > 0, 7, 3), bkv)[None]
    kv_seg = kv_seg.astype(np.int32)
    mi = oracle.mask_info(MASK_SEGMENT, 0, q_seg, kv_seg, 1, 16, nk * bkv, 16,
                          bkv)
    np.testing.assert_array_equal(mi["block_mask"][0, 0] > 0,
                                  np.asarray(valid) > 0)
    dn = mi["data_next"][0, 0]
    for step, target in printed:
        assert dn[step] == target
    for j in range(nk):
        assert valid[dn[j]] == 1          # every step lands on a valid block
        if valid[j]:
            assert dn[j] == j
    # the lists hold the valid blocks in order
    np.testing.assert_array_equal(mi["kv_idx"], np.flatnonzero(valid))


def test_data_next_trailing_and_empty_rows():
    # trailing empty steps repeat the last valid block; an empty row is 0
    q_seg = np.array([[1] * 16 + [5] * 16], dtype=np.int32)
    kv_seg = np.array([[1] * 16 + [2] * 32], dtype=np.int32)
    mi = oracle.mask_info(MASK_SEGMENT, 0, q_seg, kv_seg, 1, 32, 48, 16, 16)
    np.testing.assert_array_equal(mi["data_next"][0, 0], [0, 0, 0])
    np.testing.assert_array_equal(mi["block_mask"][0, 1], [0, 0, 0])
    np.testing.assert_array_equal(mi["data_next"][0, 1], [0, 0, 0])
    np.testing.assert_array_equal(mi["row_ptr"], [0, 1, 1])


def test_csr_lists_are_consistent():
    seg = wl.random_segment_ids(3, 700, 10, 200, 9)
    mi = oracle.mask_info(MASK_CAUSAL | MASK_SEGMENT, 0, seg, seg, 3, 700,
                          700, 64, 64)
    bm, rp = mi["block_mask"], mi["row_ptr"]
    assert bm.shape[0] == 3 and rp[-1] == len(mi["kv_idx"])
    rows = bm.reshape(-1, bm.shape[-1])
    for r in range(rows.shape[0]):
        idx = mi["kv_idx"][rp[r]:rp[r + 1]]
        np.testing.assert_array_equal(idx, np.flatnonzero(rows[r]))
        np.testing.assert_array_equal(mi["kv_cls"][rp[r]:rp[r + 1]],
                                      rows[r][idx])


def test_segment_generator_recipe():
    w = wl.WORKLOADS["cfg3_packed_s8192_d128"]
    seg = wl.make_segment_ids(w)
    assert seg.shape == (2, 8192) and seg.dtype == np.int32
    for b in range(2):
        ids = seg[b]
        assert ids[0] == 0
        d = np.diff(ids)
        assert set(np.unique(d)) <= {0, 1}
        lens = np.bincount(ids)
        assert np.all(lens[:-1] >= 256) and np.all(lens[:-1] <= 2048)
        assert 1 <= lens[-1] <= 2048
    np.testing.assert_array_equal(seg, wl.make_segment_ids(w))


@pytest.mark.parametrize("flags,window", [(1, 0), (3, 300), (5, 0), (4, 0),
                                          (7, 100), (0, 0), (2, 50)])
def test_host_flop_count_matches_oracle_pair_count(flags, window):
    # the benchmark's closed-form pair count (host logic) against the
    # oracle's element-by-element count
    from block_sparse_masked_build_gb300 import flops
    B, S = 2, 900
    seg = wl.random_segment_ids(B, S, 10, 250, 4)
    sq = seg if flags & 4 else None
    assert flops.visible_pairs(flags, window, B, S, S, sq, sq) == \
        oracle.visible_pair_count(flags, window, sq, sq, B, S, S)
    if flags & 4:  # unsorted ids take the row-by-row path
        rng = np.random.default_rng(1)
        u = rng.integers(0, 3, size=(B, S)).astype(np.int32)
        assert flops.visible_pairs(flags, window, B, S, S, u, u) == \
            oracle.visible_pair_count(flags, window, u, u, B, S, S)
