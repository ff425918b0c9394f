"""Device mask-info builder vs the oracle's brute-force scan: bit-exact."""

import numpy as np
import pytest
import torch

import oracle
import block_sparse_masked_build_gb300 as bsm
from block_sparse_masked_build_gb300 import workloads as wl
from gpu_helpers import dense_device_bits

pytestmark = pytest.mark.gpu


def _gpu_info(flags, window, seg_q, seg_kv, B, Sq, Skv, bq, bkv, dense=None,
              dense_row_words=0):
    dev = torch.device("cuda")
    qs = None if seg_q is None else torch.from_numpy(seg_q).to(dev)
    ks = None if seg_kv is None else torch.from_numpy(seg_kv).to(dev)
    db = None if dense is None else dense_device_bits(dense, dense_row_words)
    info = bsm.build_mask_info(flags, B, Sq, Skv, bq, bkv, window, qs, ks,
                               device=dev, dense_bits=db)
    torch.cuda.synchronize()
    idx, cls = info.kv_lists()
    return {
        "block_mask": info.block_mask.cpu().numpy(),
        "data_next": info.data_next.cpu().numpy(),
        "row_ptr": info.row_ptr.cpu().numpy(),
        "kv_idx": idx.cpu().numpy(),
        "kv_cls": cls.cpu().numpy(),
        "super_order": (None if info.super_order is None
                        else info.super_order.cpu().numpy()),
        "num_super": info.struct.num_super,
    }


def _check_super_order(got, ref, T, nq, bq, Sq):
    """The forward's longest-first schedule: every (table, 256-row
    super-tile) pair once, by decreasing work (rows times nonzero blocks,
    quantised to 19 bits of the largest), ties by decreasing index."""
    ns = -(-Sq // 256)
    assert got["num_super"] == ns
    order = got["super_order"]
    if T * ns > 8192:
        assert order is None
        return
    assert sorted(order.tolist()) == list(range(T * ns))
    rp = ref["row_ptr"]
    work = []
    for pr in range(T * ns):
        t, st = divmod(pr, ns)
        r0, r1 = st * 256, min(Sq, st * 256 + 256)
        w = 0
        for i in range(r0 // bq, (r1 - 1) // bq + 1):
            cnt = int(rp[t * nq + i + 1] - rp[t * nq + i])
            w += cnt * (min(r1, (i + 1) * bq) - max(r0, i * bq))
        work.append(w)
    wmax = max(max(work), 1)
    keys = [(-(w * 0x7FFFF // wmax), -i) for i, w in enumerate(work)]
    assert [-k[1] for k in sorted(keys)] == order.tolist()


def _assert_same(got, ref):
    for key in ("block_mask", "data_next", "row_ptr", "kv_idx", "kv_cls"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_mask_info_bit_exact(name):
    w = wl.WORKLOADS[name]
    seg = wl.make_segment_ids(w)
    dm = wl.make_dense_mask(w)
    ref = oracle.mask_info(w.flags, w.window, seg, seg, w.B, w.Sq, w.Skv_,
                           w.block_q, w.block_kv, dense=dm)
    got = _gpu_info(w.flags, w.window, seg, seg, w.B, w.Sq, w.Skv_, w.block_q,
                    w.block_kv, dense=dm)
    _assert_same(got, ref)
    T = w.B if w.flags & 4 else 1
    _check_super_order(got, ref, T, -(-w.Sq // w.block_q), w.block_q, w.Sq)


CASES = []
_rng = np.random.default_rng(77)
for _n in range(40):
    _flags = int(_rng.choice([0, 1, 2, 3, 4, 5, 6, 7]))
    _bq = int(_rng.choice([16, 32, 64, 128, 256]))
    _bkv = int(_rng.choice([16, 32, 64, 128, 256]))
    _Sq = int(_rng.integers(1, 700))
    _Skv = _Sq if _flags & 1 else int(_rng.integers(1, 700))
    CASES.append((_n, _flags, int(_rng.integers(1, 300)), _bq, _bkv, _Sq, _Skv,
                  int(_rng.integers(1, 4))))


@pytest.mark.parametrize("n,flags,window,bq,bkv,Sq,Skv,B", CASES)
def test_random_tiny_mask_info_bit_exact(n, flags, window, bq, bkv, Sq, Skv, B):
    rng = np.random.default_rng(1000 + n)
    seg_q = seg_kv = None
    if flags & 4:
        if n % 3 == 0:  # unsorted arbitrary ids
            seg_q = rng.integers(0, 4, size=(B, Sq)).astype(np.int32)
            seg_kv = rng.integers(0, 4, size=(B, Skv)).astype(np.int32)
        else:
            seg_q = wl.random_segment_ids(B, max(Sq, Skv), 3, 90,
                                          n)[:, :Sq].copy()
            seg_kv = wl.random_segment_ids(B, max(Sq, Skv), 3, 90,
                                           n)[:, :Skv].copy()
    ref = oracle.mask_info(flags, window, seg_q, seg_kv, B, Sq, Skv, bq, bkv)
    got = _gpu_info(flags, window, seg_q, seg_kv, B, Sq, Skv, bq, bkv)
    _assert_same(got, ref)
    T = B if flags & 4 else 1
    _check_super_order(got, ref, T, -(-Sq // bq), bq, Sq)


BAND_CASES = []
_rng_b = np.random.default_rng(78)
for _n in range(16):
    _bq = int(_rng_b.choice([16, 32, 64, 128, 256]))
    _bkv = int(_rng_b.choice([16, 32, 64, 128, 256]))
    _S = int(_rng_b.integers(1, 700))
    BAND_CASES.append((_n, 2 | 8 | (4 if _n % 4 == 3 else 0),
                       int(_rng_b.integers(1, 300)), _bq, _bkv, _S,
                       int(_rng_b.integers(1, 3))))


@pytest.mark.parametrize("n,flags,window,bq,bkv,S,B", BAND_CASES)
def test_symmetric_window_mask_info_bit_exact(n, flags, window, bq, bkv, S,
                                              B):
    seg = None
    if flags & 4:
        seg = wl.random_segment_ids(B, S, 3, 90, 500 + n)
    ref = oracle.mask_info(flags, window, seg, seg, B, S, S, bq, bkv)
    got = _gpu_info(flags, window, seg, seg, B, S, S, bq, bkv)
    _assert_same(got, ref)


DENSE_CASES = []
_rng_d = np.random.default_rng(79)
for _n in range(14):
    _bq = int(_rng_d.choice([16, 32, 64, 128]))
    _bkv = int(_rng_d.choice([16, 32, 64, 128]))
    _Sq = int(_rng_d.integers(1, 600))
    _extra = int(_rng_d.choice([0, 1, 2, 4]))  # +causal / local / segment
    _Skv = _Sq if _extra else int(_rng_d.integers(1, 600))
    DENSE_CASES.append((_n, 16 | _extra, int(_rng_d.integers(20, 200)), _bq,
                        _bkv, _Sq, _Skv, int(_rng_d.integers(1, 3))))


@pytest.mark.parametrize("n,flags,window,bq,bkv,Sq,Skv,B", DENSE_CASES)
def test_dense_mask_info_bit_exact(n, flags, window, bq, bkv, Sq, Skv, B):
    dm = wl.random_dense_mask(Sq, Skv, 0.35, int(min(bq, bkv)), 600 + n)
    seg = None
    if flags & 4:
        seg = wl.random_segment_ids(B, Sq, 3, 90, 700 + n)
    ref = oracle.mask_info(flags, window, seg, seg, B, Sq, Skv, bq, bkv,
                           dense=dm)
    got = _gpu_info(flags, window, seg, seg, B, Sq, Skv, bq, bkv, dense=dm,
                    dense_row_words=n % 3)
    _assert_same(got, ref)


@pytest.mark.parametrize("B,S,bq,bkv", [(2, 300, 32, 64), (1, 513, 64, 16)])
def test_dense_mask_with_unsorted_segments_bit_exact(B, S, bq, bkv):
    # arbitrary mask AND unsorted segment ids: the element-scan path
    rng = np.random.default_rng(S)
    seg = rng.integers(0, 3, size=(B, S)).astype(np.int32)
    dm = wl.random_dense_mask(S, S, 0.5, 32, S + 1)
    flags = 16 | 4 | 1
    ref = oracle.mask_info(flags, 0, seg, seg, B, S, S, bq, bkv, dense=dm)
    got = _gpu_info(flags, 0, seg, seg, B, S, S, bq, bkv, dense=dm)
    _assert_same(got, ref)


def test_super_order_absent_above_limit():
    # 9 tables x 1024 super-tiles exceed the 8192-pair table: no order, and
    # the forward falls back to taking the last super-tiles first
    B, Sq = 9, 262144
    seg = np.zeros((B, Sq), np.int32)
    got = _gpu_info(4, 0, seg, seg, B, Sq, 256, 512, 512)
    assert got["super_order"] is None and got["num_super"] == 1024


@pytest.mark.parametrize("S,b", [
    (65536, 64),    # 2^20 block cells: the one-launch build's largest mask
    (131072, 64),   # 2^22 cells: classify, a one-CTA scan, a compaction
    (262144, 128),  # the longest sequence the kernels take
])
def test_large_causal_mask_lists_closed_form(S, b):
    # causal classes are 2 below the diagonal, 1 on it, 0 above; each row's
    # list is its nonzero blocks in order
    got = _gpu_info(1, 0, None, None, 1, S, S, b, b)
    n = S // b
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    want = np.where(j < i, 2, np.where(j == i, 1, 0)).astype(np.int8)
    np.testing.assert_array_equal(got["block_mask"].reshape(n, n), want)
    rp = got["row_ptr"]
    np.testing.assert_array_equal(np.diff(rp), np.arange(1, n + 1))
    for r in (0, 1, 517, n // 2 + 3, n - 1):
        np.testing.assert_array_equal(got["kv_idx"][rp[r]:rp[r + 1]],
                                      np.arange(r + 1))
        np.testing.assert_array_equal(got["kv_cls"][rp[r]:rp[r + 1]],
                                      np.r_[np.full(r, 2), 1].astype(np.int8))


def test_empty_kv_mask_info():
    got = _gpu_info(0, 0, None, None, 1, 100, 0, 64, 64)
    assert got["block_mask"].shape == (1, 2, 0)
    np.testing.assert_array_equal(got["row_ptr"], [0, 0, 0])


@pytest.mark.parametrize("sorted_ids", [True, False])
def test_segment_ranges_and_sorted_flag(sorted_ids):
    B, Sq, Skv = 3, 700, 650
    if sorted_ids:
        q_seg = wl.random_segment_ids(B, 800, 5, 120, 3)[:, :Sq].copy()
        kv_seg = wl.random_segment_ids(B, 800, 5, 120, 3)[:, :Skv].copy()
    else:
        rng = np.random.default_rng(5)
        q_seg = rng.integers(0, 6, size=(B, Sq)).astype(np.int32)
        kv_seg = rng.integers(0, 6, size=(B, Skv)).astype(np.int32)
    dev = torch.device("cuda")
    info = bsm.build_mask_info(bsm.MASK_CAUSAL | bsm.MASK_SEGMENT, B, Sq, Skv,
                               64, 64, 0, torch.from_numpy(q_seg).to(dev),
                               torch.from_numpy(kv_seg).to(dev), device=dev)
    torch.cuda.synchronize()
    flag = int(info.seg_flags.cpu()[0])
    assert (flag & 1) == (0 if sorted_ids else 1)
    if sorted_ids:
        got = info.seg_range.cpu().numpy()
        for b in range(B):
            lo = np.searchsorted(kv_seg[b], q_seg[b], side="left")
            hi = np.searchsorted(kv_seg[b], q_seg[b], side="right") - 1
            np.testing.assert_array_equal(got[b, :, 0], lo)
            np.testing.assert_array_equal(got[b, :, 1], hi)


# ---- bit-packing of an arbitrary mask (the library's packing kernel)

@pytest.mark.parametrize("Sq,Skv,offset,extra_words,dtype", [
    (45, 70, 0, 0, "bool"),        # ragged last word, aligned rows
    (128, 4096, 0, 0, "bool"),     # whole words only, 16-byte loads
    (33, 97, 3, 5, "bool"),        # unaligned rows (byte loads), row padding
    (257, 1000, 16, 2, "uint8"),   # nonzero bytes other than 1 count as set
])
def test_pack_dense_mask_kernel_layout(Sq, Skv, offset, extra_words, dtype):
    """bit k % 32 of word k // 32 of row q is mask[q, k]; padding words 0."""
    m = wl.random_dense_mask(Sq, Skv, 0.5, 16, Sq + Skv)
    dev = torch.device("cuda")
    stride = Skv + offset
    raw = np.zeros(offset + Sq * stride, dtype=np.uint8)
    vals = m.astype(np.uint8)
    if dtype == "uint8":  # any nonzero byte is "visible"
        rng = np.random.default_rng(5)
        vals = vals * rng.integers(1, 256, size=m.shape, dtype=np.uint8)
    raw[offset:].reshape(Sq, stride)[:, :Skv] = vals
    buf = torch.from_numpy(raw).to(dev)
    if dtype == "bool":
        buf = buf.view(torch.bool)
    view = buf[offset:].view(Sq, stride)[:, :Skv]
    W = -(-Skv // 32) + extra_words
    words = torch.full((Sq, W), -1, dtype=torch.int32, device=dev)
    bsm.bsm_pack_dense_mask(view, words)
    torch.cuda.synchronize()
    got = words.cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, wl.pack_dense_mask(m, W))


def test_splash_attention_packs_a_dense_mask_on_the_device():
    """The end-to-end call with a boolean mask: packed by the library's
    kernel, then the forward against the oracle."""
    from gpu_helpers import compare_out, compare_lse
    B, H, Sq, Skv, D = 1, 2, 384, 448, 64
    g = torch.Generator().manual_seed(77)
    q = torch.randn(B, H, Sq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, Skv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, Skv, D, generator=g).to(torch.bfloat16)
    m = wl.random_dense_mask(Sq, Skv, 0.4, 64, 78)
    dev = torch.device("cuda")
    out, lse = bsm.splash_attention(
        q.to(dev), k.to(dev), v.to(dev), mask_flags=bsm.MASK_DENSE,
        dense_mask=torch.from_numpy(m).to(dev))
    torch.cuda.synchronize()
    scale = 1.0 / np.sqrt(D)
    ref, ref_lse = oracle.softmax_attention(q, k, v, bsm.MASK_DENSE, 0, None,
                                            None, scale, dense=m)
    compare_out(out.float().cpu().numpy(), ref, what="dense out")
    compare_lse(lse.cpu().numpy(), ref_lse, what="dense lse")
