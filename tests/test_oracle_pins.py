"""Pins of the fp64 oracle's attention arithmetic against facts outside it.

Each test checks the oracle against something it does not compute itself:
an invariant the splash notes state (weights sum to one, causal row 0), a
library routine in a special case (torch's scaled_dot_product_attention and
silu in float64, scipy's logsumexp) with masks built here by a different
construction (np.tril / block-diagonal segments), the online recurrence of
the splash notes section 15 (which must give the two-pass result for any
block size), and scalar closed forms evaluated with ``math``.
"""

import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from oracle import MASK_CAUSAL, MASK_LOCAL, MASK_SEGMENT
from block_sparse_masked_build_gb300 import workloads as wl


def _qkv(B, H, Sq, Skv, D, seed, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, D, generator=g) * sigma).to(torch.bfloat16)
    k = (torch.randn(B, H, Skv, D, generator=g) * sigma).to(torch.bfloat16)
    v = (torch.randn(B, H, Skv, D, generator=g) * sigma).to(torch.bfloat16)
    return q, k, v


def _segments_from_lengths(lens):
    return np.repeat(np.arange(len(lens), dtype=np.int32), lens)


def _block_diag_mask(lens):
    """Same-segment mask built from segment lengths with np.kron-free loops."""
    S = sum(lens)
    m = np.zeros((S, S), dtype=bool)
    o = 0
    for n in lens:
        m[o:o + n, o:o + n] = True
        o += n
    return m


def _sdpa64(q, k, v, mask, scale):
    qq = q.to(torch.float64)
    kk = k.to(torch.float64)
    vv = v.to(torch.float64)
    return torch.nn.functional.scaled_dot_product_attention(
        qq, kk, vv, attn_mask=torch.from_numpy(mask), scale=scale).numpy()


MASKS = [
    (0, 0),
    (MASK_CAUSAL, 0),
    (MASK_CAUSAL | MASK_LOCAL, 37),
    (MASK_CAUSAL | MASK_SEGMENT, 0),
    (MASK_SEGMENT, 0),
    (MASK_LOCAL, 20),
]


@pytest.mark.parametrize("flags,window", MASKS)
def test_constant_value_rows_give_that_row(flags, window):
    # splash notes 15.3: Out = O / L, a weighted mean of the v rows whose
    # weights add up to one; with every v row equal to c the output is c.
    B, H, S, D = 2, 2, 160, 32
    q, k, _ = _qkv(B, H, S, S, D, 11)
    c = torch.linspace(-2, 3, D).to(torch.bfloat16)
    v = c.expand(B, H, S, D).clone()
    seg = wl.random_segment_ids(B, S, 5, 40, 3)
    out, lse = oracle.softmax_attention(q, k, v, flags, window, seg, seg,
                                        0.17)
    np.testing.assert_allclose(out, np.broadcast_to(
        c.double().numpy(), out.shape), rtol=0, atol=1e-12)
    assert np.all(np.isfinite(lse))


@pytest.mark.parametrize("flags", [MASK_CAUSAL, MASK_CAUSAL | MASK_LOCAL,
                                   MASK_CAUSAL | MASK_SEGMENT])
def test_causal_row0_returns_v0(flags):
    # Causal row 0 sees only key 0: out = v_0 and lse = scale * q_0 . k_0.
    B, H, S, D = 1, 3, 96, 64
    q, k, v = _qkv(B, H, S, S, D, 12)
    seg = wl.random_segment_ids(B, S, 8, 30, 4)
    scale = 1 / 8
    out, lse = oracle.softmax_attention(q, k, v, flags, 50, seg, seg, scale)
    for h in range(H):
        np.testing.assert_allclose(out[0, h, 0], v[0, h, 0].double().numpy(),
                                   rtol=0, atol=1e-12)
        dot = math.fsum(float(a) * float(b) for a, b in
                        zip(q[0, h, 0].tolist(), k[0, h, 0].tolist()))
        assert abs(lse[0, h, 0] - scale * dot) < 1e-10


def test_full_mask_matches_torch_sdpa_fp64():
    B, H, Sq, Skv, D = 2, 3, 70, 90, 64
    q, k, v = _qkv(B, H, Sq, Skv, D, 13)
    out, _ = oracle.softmax_attention(q, k, v, 0, 0, None, None, 0.125)
    ref = _sdpa64(q, k, v, np.ones((Sq, Skv), dtype=bool), 0.125)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_causal_matches_torch_sdpa_fp64():
    B, H, S, D = 1, 2, 130, 32
    q, k, v = _qkv(B, H, S, S, D, 14)
    out, _ = oracle.softmax_attention(q, k, v, MASK_CAUSAL, 0, None, None,
                                      0.3)
    ref = _sdpa64(q, k, v, np.tril(np.ones((S, S), dtype=bool)), 0.3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_local_window_matches_sdpa_band_mask():
    # causal AND q - k < W  ==  lower band of width W (np.tril/np.triu).
    B, H, S, D, W = 1, 2, 150, 32, 23
    q, k, v = _qkv(B, H, S, S, D, 15)
    out, _ = oracle.softmax_attention(q, k, v, MASK_CAUSAL | MASK_LOCAL, W,
                                      None, None, 0.2)
    ones = np.ones((S, S), dtype=bool)
    band = np.tril(ones) & np.triu(ones, -(W - 1))
    ref = _sdpa64(q, k, v, band, 0.2)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_symmetric_window_matches_sdpa_band_mask():
    # |q - k| < W  ==  np.triu(., -(W-1)) & np.tril(., W-1)
    B, H, S, D, W = 1, 2, 150, 32, 23
    q, k, v = _qkv(B, H, S, S, D, 16)
    flags = oracle.MASK_LOCAL | oracle.MASK_BAND
    out, _ = oracle.softmax_attention(q, k, v, flags, W, None, None, 0.2)
    ones = np.ones((S, S), dtype=bool)
    band = np.tril(ones, W - 1) & np.triu(ones, -(W - 1))
    ref = _sdpa64(q, k, v, band, 0.2)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_dense_mask_matches_sdpa_with_that_mask():
    # an arbitrary mask: the oracle equals float64 SDPA given the same
    # boolean matrix (rows kept non-empty so SDPA stays defined)
    from block_sparse_masked_build_gb300 import workloads as wl
    B, H, S, D = 1, 2, 130, 32
    q, k, v = _qkv(B, H, S, S, D, 19)
    dm = wl.random_dense_mask(S, S, 0.3, 32, 20)
    dm[np.arange(S), np.arange(S)] = True
    out, _ = oracle.softmax_attention(q, k, v, oracle.MASK_DENSE, 0, None,
                                      None, 0.2, dense=dm)
    np.testing.assert_allclose(out, _sdpa64(q, k, v, dm, 0.2), rtol=0,
                               atol=1e-12)


def test_dense_mask_special_cases():
    # all-true dense mask changes nothing; a lower-triangular one is causal
    B, H, S, D = 1, 1, 90, 16
    q, k, v = _qkv(B, H, S, S, D, 21)
    ones = np.ones((S, S), dtype=bool)
    a, la = oracle.softmax_attention(q, k, v, oracle.MASK_DENSE, 0, None,
                                     None, 0.3, dense=ones)
    b, lb = oracle.softmax_attention(q, k, v, 0, 0, None, None, 0.3)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    c, lc = oracle.softmax_attention(q, k, v, oracle.MASK_DENSE, 0, None,
                                     None, 0.3, dense=np.tril(ones))
    d, ld = oracle.softmax_attention(q, k, v, MASK_CAUSAL, 0, None, None, 0.3)
    np.testing.assert_array_equal(c, d)
    np.testing.assert_array_equal(lc, ld)


def test_packed_segments_match_sdpa_block_diagonal_mask():
    B, H, D = 1, 2, 32
    lens = [17, 40, 3, 60, 30]
    S = sum(lens)
    q, k, v = _qkv(B, H, S, S, D, 16)
    seg = _segments_from_lengths(lens)[None]
    out, lse = oracle.softmax_attention(q, k, v, MASK_CAUSAL | MASK_SEGMENT, 0,
                                        seg, seg, 0.25)
    mask = _block_diag_mask(lens) & np.tril(np.ones((S, S), dtype=bool))
    ref = _sdpa64(q, k, v, mask, 0.25)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # lse against scipy's logsumexp over the same visible scores
    s = 0.25 * (q[0, 0].double() @ k[0, 0].double().T).numpy()
    s = np.where(mask, s, -np.inf)
    np.testing.assert_allclose(lse[0, 0], logsumexp(s, axis=1), rtol=0,
                               atol=1e-12)


@pytest.mark.parametrize("block", [1, 7, 16, 64, 200])
@pytest.mark.parametrize("flags,window", MASKS)
def test_online_recurrence_equals_two_pass(block, flags, window):
    # splash notes 15.1-15.3: streaming over KV blocks with m, l, o and the
    # correction alpha gives the same Out (and lse) for every block size.
    B, H, Sq, Skv, D = 1, 1, 120, 120, 16
    q, k, v = _qkv(B, H, Sq, Skv, D, 17)
    seg = wl.random_segment_ids(B, Sq, 3, 25, 5)
    out2, lse2 = oracle.softmax_attention(q, k, v, flags, window, seg, seg,
                                          0.4)
    out1, lse1 = oracle.softmax_attention_online(q, k, v, flags, window, seg,
                                                 seg, 0.4, block)
    np.testing.assert_allclose(out1, out2[0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse2[0, 0], rtol=0, atol=1e-12)


def test_fully_masked_row_gives_zero_and_neg_inf():
    # q segment 9 exists in no kv position: every element of those rows is
    # masked.
    B, H, S, D = 1, 1, 64, 16
    q, k, v = _qkv(B, H, S, S, D, 18)
    qseg = np.zeros((1, S), dtype=np.int32)
    qseg[0, 10:20] = 9
    kvseg = np.zeros((1, S), dtype=np.int32)
    out, lse = oracle.softmax_attention(q, k, v, MASK_SEGMENT, 0, qseg, kvseg,
                                        0.3)
    assert np.all(out[0, 0, 10:20] == 0)
    assert np.all(np.isneginf(lse[0, 0, 10:20]))
    assert np.all(np.isfinite(lse[0, 0, :10]))
    out_p = oracle.pointwise_attention(q, k, v, MASK_SEGMENT, 0, qseg, kvseg,
                                       0.3)
    assert np.all(out_p[0, 0, 10:20] == 0)


def test_rows_api_matches_full_api():
    B, H, S, D = 2, 2, 100, 32
    q, k, v = _qkv(B, H, S, S, D, 19)
    seg = wl.random_segment_ids(B, S, 5, 30, 6)
    fl = MASK_CAUSAL | MASK_SEGMENT
    out, lse = oracle.softmax_attention(q, k, v, fl, 0, seg, seg, 0.3)
    rows = [(1, 0, 99), (0, 1, 0), (0, 1, 57), (1, 1, 3)]
    o2, l2 = oracle.softmax_attention(q, k, v, fl, 0, seg, seg, 0.3, rows=rows)
    # equal up to the summation order of the matrix product
    for n, (b, h, r) in enumerate(rows):
        np.testing.assert_allclose(o2[n], out[b, h, r], rtol=0, atol=1e-13)
        assert abs(l2[n] - lse[b, h, r]) < 1e-13
    p = oracle.pointwise_attention(q, k, v, fl, 0, seg, seg, 0.3)
    p2 = oracle.pointwise_attention(q, k, v, fl, 0, seg, seg, 0.3, rows=rows)
    for n, (b, h, r) in enumerate(rows):
        np.testing.assert_allclose(p2[n], p[b, h, r], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- pointwise

def test_pointwise_row0_closed_form():
    # hstu_ops fwd: p = x * logistic(x) / seq_len with x = scale * q.k;
    # causal row 0 sees only key 0, so out_0 = p_00 * v_0.
    B, H, S, D = 1, 2, 64, 32
    q, k, v = _qkv(B, H, S, S, D, 20, sigma=0.5)
    scale = 0.7
    out = oracle.pointwise_attention(q, k, v, MASK_CAUSAL, 0, None, None,
                                     scale)
    for h in range(H):
        dot = math.fsum(float(a) * float(b) for a, b in
                        zip(q[0, h, 0].tolist(), k[0, h, 0].tolist()))
        x = scale * dot
        p = x / (1.0 + math.exp(-x)) / S
        np.testing.assert_allclose(out[0, h, 0], p * v[0, h, 0].double().numpy(),
                                   rtol=1e-13, atol=1e-15)


def test_pointwise_full_mask_matches_torch_silu():
    B, H, Sq, Skv, D = 2, 2, 48, 80, 32
    q, k, v = _qkv(B, H, Sq, Skv, D, 21)
    scale = 0.3
    out = oracle.pointwise_attention(q, k, v, 0, 0, None, None, scale)
    x = scale * (q.double() @ k.double().transpose(-1, -2))
    ref = (torch.nn.functional.silu(x) / Sq) @ v.double()
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-13)


def test_pointwise_causal_matches_torch_tril():
    B, H, S, D = 1, 2, 90, 32
    q, k, v = _qkv(B, H, S, S, D, 22)
    out = oracle.pointwise_attention(q, k, v, MASK_CAUSAL, 0, None, None, 0.2)
    x = 0.2 * (q.double() @ k.double().transpose(-1, -2))
    p = torch.nn.functional.silu(x) / S
    p = torch.tril(p)
    np.testing.assert_allclose(out, (p @ v.double()).numpy(), rtol=0,
                               atol=1e-13)


def test_pointwise_is_linear_in_v():
    B, H, S, D = 1, 1, 70, 16
    q, k, v1 = _qkv(B, H, S, S, D, 23)
    _, _, v2 = _qkv(B, H, S, S, D, 24)
    seg = wl.random_segment_ids(B, S, 5, 20, 7)
    fl = MASK_CAUSAL | MASK_SEGMENT
    a, b = 0.75, -2.0
    v12 = (a * v1.double() + b * v2.double())
    o1 = oracle.pointwise_attention(q, k, v1, fl, 0, seg, seg, 0.5)
    o2 = oracle.pointwise_attention(q, k, v2, fl, 0, seg, seg, 0.5)
    o12 = oracle.pointwise_attention(q, k, v12, fl, 0, seg, seg, 0.5)
    np.testing.assert_allclose(o12, a * o1 + b * o2, rtol=0, atol=1e-13)


def test_pointwise_uses_query_length_not_key_length():
    # hstu_ops passes seq_len = q_seq_len to the forward kernel: doubling the
    # keys with an exact copy (full mask) doubles the output.
    B, H, Sq, D = 1, 1, 32, 16
    q, k, v = _qkv(B, H, Sq, 40, D, 25)
    k2 = torch.cat([k, k], dim=2)
    v2 = torch.cat([v, v], dim=2)
    o1 = oracle.pointwise_attention(q, k, v, 0, 0, None, None, 0.3)
    o2 = oracle.pointwise_attention(q, k2, v2, 0, 0, None, None, 0.3)
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-13, atol=1e-15)


def test_pointwise_under_band_and_dense_masks():
    # the pointwise path under the extra masks: an all-true arbitrary mask
    # is the full mask, a lower-triangular one is causal, and the symmetric
    # window equals the same band given as an arbitrary mask
    B, H, S, D = 1, 2, 80, 16
    q, k, v = _qkv(B, H, S, S, D, 27, sigma=0.5)
    ones = np.ones((S, S), dtype=bool)
    dn = oracle.MASK_DENSE
    a = oracle.pointwise_attention(q, k, v, dn, 0, None, None, 0.3,
                                   dense=ones)
    np.testing.assert_array_equal(
        a, oracle.pointwise_attention(q, k, v, 0, 0, None, None, 0.3))
    c = oracle.pointwise_attention(q, k, v, dn, 0, None, None, 0.3,
                                   dense=np.tril(ones))
    np.testing.assert_array_equal(
        c, oracle.pointwise_attention(q, k, v, MASK_CAUSAL, 0, None, None,
                                      0.3))
    W = 7
    band = np.tril(ones, W - 1) & np.triu(ones, -(W - 1))
    e = oracle.pointwise_attention(q, k, v, MASK_LOCAL | oracle.MASK_BAND, W,
                                   None, None, 0.3)
    np.testing.assert_array_equal(
        e, oracle.pointwise_attention(q, k, v, dn, 0, None, None, 0.3,
                                      dense=band))
