"""Host-side work accounting: visible (q, k) pairs and unmasked FLOPs.

Unmasked FLOPs count 4*D per visible pair (2*D for q.k, 2*D for p*v); exp,
masking, rescaling and masked slots inside partial tiles are not counted.
Counts are per-row closed forms: row q sees keys in
[max(0, q-window+1, seg_start(q)), min(q, Skv-1)] under causal/local/
(sorted, contiguous) segment masks; other segment-id arrays are counted by
comparing ids row by row.
"""

from __future__ import annotations

import numpy as np

MASK_CAUSAL = 1
MASK_LOCAL = 2
MASK_SEGMENT = 4
MASK_BAND = 8
MASK_DENSE = 16


def _rows_range(flags, window, Sq, Skv):
    q = np.arange(Sq, dtype=np.int64)
    lo = np.zeros(Sq, dtype=np.int64)
    hi = np.full(Sq, Skv - 1, dtype=np.int64)
    if flags & MASK_CAUSAL:
        hi = np.minimum(hi, q)
    if flags & MASK_LOCAL:  # q - k < window
        lo = np.maximum(lo, q - window + 1)
    if flags & MASK_BAND:  # and k - q < window
        hi = np.minimum(hi, q + window - 1)
    return lo, hi


def _dense_rows(flags, window, Sq, Skv, q_seg, kv_seg, dense, slab=1024):
    """Visible keys per row with an arbitrary mask: the mask's set bits
    inside each row's key range (and segment), counted in row slabs."""
    lo, hi = _rows_range(flags, window, Sq, Skv)
    dense = np.asarray(dense, dtype=bool)
    k = np.arange(Skv)
    out = np.zeros(Sq, dtype=np.int64)
    for r0 in range(0, Sq, slab):
        r = np.arange(r0, min(Sq, r0 + slab))
        m = dense[r] & (k[None, :] >= lo[r, None]) & (k[None, :] <= hi[r, None])
        if flags & MASK_SEGMENT:
            m &= np.asarray(kv_seg)[None, :] == np.asarray(q_seg)[r, None]
        out[r] = m.sum(axis=1)
    return out


def visible_pairs_per_row(flags, window, Sq, Skv, q_seg=None, kv_seg=None,
                          dense=None):
    """int64 [Sq] visible keys per query row for one batch row."""
    if flags & MASK_DENSE:
        return _dense_rows(flags, window, Sq, Skv, q_seg, kv_seg, dense)
    lo, hi = _rows_range(flags, window, Sq, Skv)
    if not (flags & MASK_SEGMENT):
        return np.maximum(0, hi - lo + 1)
    q_seg = np.asarray(q_seg)
    kv_seg = np.asarray(kv_seg)
    same = (Sq == Skv) and np.array_equal(q_seg, kv_seg)
    if same and np.all(np.diff(kv_seg) >= 0):
        # contiguous segments: a row sees keys from its segment's start on
        first = np.searchsorted(kv_seg, q_seg, side="left")
        last = np.searchsorted(kv_seg, q_seg, side="right") - 1
        lo2 = np.maximum(lo, first)
        hi2 = np.minimum(hi, last)
        return np.maximum(0, hi2 - lo2 + 1)
    out = np.zeros(Sq, dtype=np.int64)
    for r in range(Sq):
        if hi[r] >= lo[r]:
            out[r] = int(np.count_nonzero(kv_seg[lo[r]:hi[r] + 1] == q_seg[r]))
    return out


def visible_pairs(flags, window, B, Sq, Skv, q_seg=None, kv_seg=None,
                  dense=None):
    """Visible pairs summed over batch rows (one head)."""
    if not (flags & MASK_SEGMENT):
        return int(B * visible_pairs_per_row(flags, window, Sq, Skv,
                                             dense=dense).sum())
    return int(sum(visible_pairs_per_row(flags, window, Sq, Skv, q_seg[b],
                                         kv_seg[b], dense).sum()
                   for b in range(B)))


def unmasked_flops(flags, window, B, H, Sq, Skv, D, q_seg=None, kv_seg=None,
                   dense=None):
    return 4 * D * H * visible_pairs(flags, window, B, Sq, Skv, q_seg, kv_seg,
                                     dense)
