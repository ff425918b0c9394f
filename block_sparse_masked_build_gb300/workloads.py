"""Seeded synthetic inputs for block-sparse masked attention.

This module only draws inputs: it holds none of the attention arithmetic and
imports nothing else from this package, so that both the CUDA path and the
fp64 oracle can be fed from it without sharing any computation.

Workloads follow the five shapes the attention-forward study defines
(causal softmax MHA at small and medium size, packed sequences with segment
ids, HSTU pointwise attention, and a long local-window mask), plus two
diagnostic variants: the packed-sequence shape with the segment mask switched
off ("3c"), and the HSTU shape with scale 1/sqrt(D) ("4p") whose outputs are
large enough for absolute tolerances to mean something.

Input recipe:
  * q, k, v: drawn in that order from one CPU ``torch.Generator`` seeded with
    the workload's seed, as float32 normal(0, 1) times ``sigma``, then rounded
    to bfloat16 (round-to-nearest-even), layout [B, H, S, D] contiguous.
  * segment ids: per batch row, ``numpy.random.default_rng(seed)`` draws
    integer lengths uniform in [seg_min, seg_max] (inclusive) until they cover
    S; the last segment is truncated; ids are 0, 1, 2, ... in order; the
    q and kv ids are the same array.
"""

from __future__ import annotations

import dataclasses
import functools
import math

import numpy as np
import torch

# Mask predicate flags (same bit values as the C interface).
MASK_CAUSAL = 1
MASK_LOCAL = 2
MASK_SEGMENT = 4
MASK_BAND = 8
MASK_DENSE = 16

SCORE_SOFTMAX = 0
SCORE_POINTWISE = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    block_q: int
    block_kv: int
    flags: int
    window: int
    score: int
    scale: float
    sigma: float
    seed: int
    seg_min: int = 256
    seg_max: int = 2048
    Skv: int | None = None  # None: same as S
    dense_p: float = 0.5    # MASK_DENSE: P(visible) inside random tiles
    Hkv: int | None = None  # K/V heads (None: H); H must be a multiple

    @property
    def Sq(self) -> int:
        return self.S

    @property
    def Skv_(self) -> int:
        return self.S if self.Skv is None else self.Skv

    @property
    def Hkv_(self) -> int:
        return self.H if self.Hkv is None else self.Hkv

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    # causal softmax, B=1 H=2 S=256 D=64, 64x64 blocks (the small case)
    "cfg1_causal_s256_d64": Workload(
        "cfg1_causal_s256_d64", 1, 2, 256, 64, 64, 64, MASK_CAUSAL, 0,
        SCORE_SOFTMAX, 1.0 / math.sqrt(64), 1.0, 1001),
    # causal softmax, B=4 H=16 S=2048 D=128
    "cfg2_causal_s2048_d128": Workload(
        "cfg2_causal_s2048_d128", 4, 16, 2048, 128, 128, 128, MASK_CAUSAL, 0,
        SCORE_SOFTMAX, 1.0 / math.sqrt(128), 1.0, 1002),
    # packed sequences: causal AND same-segment, B=2 H=16 S=8192 D=128
    "cfg3_packed_s8192_d128": Workload(
        "cfg3_packed_s8192_d128", 2, 16, 8192, 128, 128, 128,
        MASK_CAUSAL | MASK_SEGMENT, 0, SCORE_SOFTMAX, 1.0 / math.sqrt(128),
        1.0, 1003),
    # the same shapes and seed with the segment mask off (pure causal)
    "cfg3c_causal_s8192_d128": Workload(
        "cfg3c_causal_s8192_d128", 2, 16, 8192, 128, 128, 128, MASK_CAUSAL, 0,
        SCORE_SOFTMAX, 1.0 / math.sqrt(128), 1.0, 1003),
    # HSTU pointwise, causal, B=16 H=8 S=4096 D=128, N(0, 0.5), scale = 1/S
    "cfg4_hstu_s4096_d128": Workload(
        "cfg4_hstu_s4096_d128", 16, 8, 4096, 128, 128, 128, MASK_CAUSAL, 0,
        SCORE_POINTWISE, 1.0 / 4096, 0.5, 1004),
    # HSTU pointwise with scale 1/sqrt(D) (parity-only variant)
    "cfg4p_hstu_s4096_d128": Workload(
        "cfg4p_hstu_s4096_d128", 16, 8, 4096, 128, 128, 128, MASK_CAUSAL, 0,
        SCORE_POINTWISE, 1.0 / math.sqrt(128), 0.5, 1004),
    # local window: causal AND q-k < 4096, B=1 H=32 S=32768 D=128
    "cfg5_local_s32768_d128": Workload(
        "cfg5_local_s32768_d128", 1, 32, 32768, 128, 128, 128,
        MASK_CAUSAL | MASK_LOCAL, 4096, SCORE_SOFTMAX, 1.0 / math.sqrt(128),
        1.0, 1005),
    # beyond the five workloads, diagnostics of the extensions:
    # symmetric sliding window |q - k| < 1024, B=2 H=16 S=8192 D=128
    "next3_band_s8192_d128": Workload(
        "next3_band_s8192_d128", 2, 16, 8192, 128, 128, 128,
        MASK_LOCAL | MASK_BAND, 1024, SCORE_SOFTMAX, 1.0 / math.sqrt(128),
        1.0, 1006),
    # an arbitrary mask AND causal (128-square tiles empty, full or random
    # with P = 0.5), B=2 H=16 S=8192 D=128
    "next2_dense_s8192_d128": Workload(
        "next2_dense_s8192_d128", 2, 16, 8192, 128, 128, 128,
        MASK_DENSE | MASK_CAUSAL, 0, SCORE_SOFTMAX, 1.0 / math.sqrt(128), 1.0,
        1007),
    # grouped-query attention: 32 query heads over 8 K/V heads, causal,
    # B=2 S=8192 D=128
    "next1_gqa_s8192_d128": Workload(
        "next1_gqa_s8192_d128", 2, 32, 8192, 128, 128, 128, MASK_CAUSAL, 0,
        SCORE_SOFTMAX, 1.0 / math.sqrt(128), 1.0, 1008, Hkv=8),
}

# The configuration the headline throughput is quoted on (causal, S=8192,
# D=128, packed segments).
HEADLINE = "cfg3_packed_s8192_d128"


def make_qkv(w: Workload, B: int | None = None, H: int | None = None):
    """q [B, H, Sq, D], k and v [B, H_kv, Skv, D] as CPU bfloat16 tensors
    (contiguous).

    ``B``/``H`` may be reduced to draw a prefix-shaped sample; the values of
    the full-size draw are not reproduced in that case (the generator stream
    is consumed in a different order), so callers that compare against a
    full-size run must use the full shape.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    Hkv = H * w.Hkv_ // w.H  # K/V heads in the same ratio
    q = (torch.randn((B, H, w.Sq, w.D), generator=g, dtype=torch.float32)
         * w.sigma).to(torch.bfloat16)
    k = (torch.randn((B, Hkv, w.Skv_, w.D), generator=g, dtype=torch.float32)
         * w.sigma).to(torch.bfloat16)
    v = (torch.randn((B, Hkv, w.Skv_, w.D), generator=g, dtype=torch.float32)
         * w.sigma).to(torch.bfloat16)
    return q, k, v


def segment_lengths(rng: np.random.Generator, S: int, lo: int, hi: int):
    """Consecutive segment lengths uniform in [lo, hi], last one truncated."""
    lens = []
    total = 0
    while total < S:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, S - total)
        lens.append(n)
        total += n
    return lens


def make_segment_ids(w: Workload, B: int | None = None) -> np.ndarray | None:
    """int32 [B, S] segment ids (q and kv share them), or None if unused."""
    if not (w.flags & MASK_SEGMENT):
        return None
    B = w.B if B is None else B
    rng = np.random.default_rng(w.seed)
    out = np.empty((B, w.S), dtype=np.int32)
    for b in range(B):
        lens = segment_lengths(rng, w.S, w.seg_min, w.seg_max)
        out[b] = np.repeat(np.arange(len(lens), dtype=np.int32), lens)
    return out


def random_segment_ids(B: int, S: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Segment ids with arbitrary (small) segment lengths, for edge cases."""
    rng = np.random.default_rng(seed)
    out = np.empty((B, S), dtype=np.int32)
    for b in range(B):
        lens = segment_lengths(rng, S, lo, hi)
        out[b] = np.repeat(np.arange(len(lens), dtype=np.int32), lens)
    return out


def sample_rows(w: Workload, n: int, seed: int, seg: np.ndarray | None = None):
    """Seeded sample of (b, h, q) output rows for full-size parity checks.

    Always contains row 0, the last row, every 128-row block boundary that the
    sample budget allows, and segment starts when segment ids are given.
    """
    rng = np.random.default_rng(seed)
    rows = set()
    S = w.Sq
    must = {0, S - 1}
    for blk in (64, 128):
        for s in range(0, S, blk):
            must.add(s)
            must.add(min(S - 1, s + blk - 1))
    if seg is not None:
        starts = np.flatnonzero(np.diff(seg[0])) + 1
        must.update(int(x) for x in starts)
    must = sorted(must)
    picks = []
    for q in must:
        picks.append((int(rng.integers(w.B)), int(rng.integers(w.H)), q))
    while len(picks) < n:
        picks.append((int(rng.integers(w.B)), int(rng.integers(w.H)),
                      int(rng.integers(S))))
    for p in picks:
        rows.add(p)
    return sorted(rows)


def random_dense_mask(Sq: int, Skv: int, p_visible: float, block: int,
                      seed: int) -> np.ndarray:
    """Seeded boolean [Sq, Skv] mask for the arbitrary-mask path: each
    block x block tile is empty, full or random (visible with probability
    p_visible) with equal odds, so every block class occurs."""
    rng = np.random.default_rng(seed)
    m = rng.random((Sq, Skv)) < p_visible
    nq, nk = -(-Sq // block), -(-Skv // block)
    kind = rng.integers(0, 3, size=(nq, nk))
    for i in range(nq):
        for j in range(nk):
            sl = (slice(i * block, (i + 1) * block),
                  slice(j * block, (j + 1) * block))
            if kind[i, j] == 0:
                m[sl] = False
            elif kind[i, j] == 1:
                m[sl] = True
    return m


def pack_dense_mask(mask: np.ndarray, row_words: int = 0) -> np.ndarray:
    """Bit-pack a boolean [Sq, Skv] mask into uint32 words, row-major: bit
    k % 32 of word k // 32 of row q is mask[q, k].  row_words (>= the
    minimum ceil(Skv / 32)) pads each row."""
    Sq, Skv = mask.shape
    w = max(row_words, -(-Skv // 32))
    padded = np.zeros((Sq, w * 32), dtype=bool)
    padded[:, :Skv] = mask
    packed = np.packbits(padded, axis=1, bitorder="little")  # [Sq, 4w] bytes
    return np.ascontiguousarray(packed).view("<u4").astype(np.uint32)


@functools.lru_cache(maxsize=4)
def _dense_cached(w: Workload) -> np.ndarray:
    return random_dense_mask(w.Sq, w.Skv_, w.dense_p, w.block_q, w.seed + 100)


def make_dense_mask(w: Workload) -> np.ndarray | None:
    """The workload's boolean [Sq, Skv] arbitrary mask (MASK_DENSE), or
    None.  The same array is returned on every call: do not modify it."""
    if not (w.flags & MASK_DENSE):
        return None
    return _dense_cached(w)
