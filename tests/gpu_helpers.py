"""Shared helpers of the GPU parity tests (run the CUDA path, compare)."""

from __future__ import annotations

import numpy as np
import torch

import block_sparse_masked_build_gb300 as bsm
from block_sparse_masked_build_gb300 import workloads as wl

# Tolerances of the forward output (bf16) and the logsumexp (f32): max-abs
# 2e-2 and mean-abs 2e-3 on outputs, 1e-3 relative on logsumexp.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_REL = 1e-3
# The pointwise path's outputs are ~1e-3 (or ~1e-6 with scale = 1/S), where
# absolute gates say nothing, so it is also gated relative to the oracle's
# magnitude: max error <= 2e-2 * max|ref| and mean error <= 2e-3 * mean|ref|
# (the same 2e-2 / 2e-3 figures, relative).  hstu_ops' forward multiplies
# f32 scores by f32 v; the kernel keeps p as a bf16 pair (hi + lo, about 16
# bits), so only the bf16 output rounding remains.  test_pointwise_rounding
# emulates exactly these roundings from the oracle's values and finds
# ~1.4e-3, inside the gate; a single bf16 p would give ~2.3e-3.
PW_MAX_REL = 2e-2
PW_MEAN_REL = 2e-3
# Gradients (dQ, dK, dV) are gated relative to the reference's magnitude:
# max error <= 2e-2 * max|ref|, mean error <= 4e-3 * mean|ref|.  The
# backward rounds P and dS to bf16 (as hstu_ops' backward does) and its
# outputs to bf16; test_bwd_rounding applies exactly those roundings to the
# oracle's values and finds ~2.3e-3 relative mean error.
BWD_MAX_REL = 2e-2
BWD_MEAN_REL = 4e-3


def compare_grad(got, ref, what=""):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    err = np.abs(g - r)
    mx = max(float(np.abs(r).max()), 1e-30)
    mn = max(float(np.abs(r).mean()), 1e-30)
    assert err.max() / mx <= BWD_MAX_REL, f"{what}: rel max {err.max() / mx}"
    assert err.mean() / mn <= BWD_MEAN_REL, \
        f"{what}: rel mean {err.mean() / mn}"
    return err.max() / mx, err.mean() / mn


def dense_device_bits(dense, row_words=0):
    """Bit-packed device copy of a boolean [Sq, Skv] mask (int32 view)."""
    words = wl.pack_dense_mask(np.asarray(dense, dtype=bool), row_words)
    return torch.from_numpy(words.view(np.int32)).to("cuda")


def run_gpu(q, k, v, flags, window, q_seg, kv_seg, scale, score,
            block_q=128, block_kv=128, layout="bhsd", longest_first=True,
            dense=None, dense_row_words=0):
    """Run mask-info build + forward on the GPU; returns CPU out, lse, info.
    longest_first=False drops the mask info's unit order, so the forward
    takes its fallback schedule."""
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if layout == "bshd":  # store as [B, S, H, D] and pass transposed views
        qd = qd.transpose(1, 2).contiguous().transpose(1, 2)
        kd = kd.transpose(1, 2).contiguous().transpose(1, 2)
        vd = vd.transpose(1, 2).contiguous().transpose(1, 2)
    qs = None if q_seg is None else torch.from_numpy(np.ascontiguousarray(q_seg)).to(dev)
    ks = None if kv_seg is None else torch.from_numpy(np.ascontiguousarray(kv_seg)).to(dev)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    db = None if dense is None else dense_device_bits(dense, dense_row_words)
    info = bsm.build_mask_info(flags, B, Sq, Skv, block_q, block_kv, window,
                               qs, ks, device=dev, dense_bits=db)
    out = torch.full((B, H, Sq, D), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    if layout == "bshd":
        out = out.transpose(1, 2).contiguous().transpose(1, 2)
    lse = None
    if score == bsm.SCORE_SOFTMAX:
        lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32,
                         device=dev)
    if not longest_first:
        info.struct.super_order = None
    bsm.bsm_splash_fwd(qd, kd, vd, info, qs, ks, scale, score, out, lse)
    torch.cuda.synchronize()
    st, detail = bsm.bsm_device_status()
    assert st == 0, f"device status {st} {detail}"
    return (out.float().cpu(), None if lse is None else lse.cpu(), info)


def compare_out(got, ref, pointwise=False, what=""):
    """Max/mean absolute error gates (relative to the oracle's magnitude for
    the pointwise path, whose outputs are far below 1)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    if pointwise:
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, what
        mx = max(float(np.abs(r).max()), 1e-30)
        mn = max(float(np.abs(r).mean()), 1e-30)
        assert err.max() / mx <= PW_MAX_REL, f"{what}: rel max {err.max() / mx}"
        assert err.mean() / mn <= PW_MEAN_REL, \
            f"{what}: rel mean {err.mean() / mn}"
        return err.max() / mx, err.mean() / mn
    assert err.max() <= MAX_ABS, f"{what}: max abs {err.max()}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs {err.mean()}"
    return err.max(), err.mean()


def compare_lse(got, ref, what=""):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    inf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), inf), f"{what}: -inf rows differ"
    rel = np.abs(g[~inf] - r[~inf]) / np.maximum(1.0, np.abs(r[~inf]))
    if rel.size:
        assert rel.max() <= LSE_REL, f"{what}: lse rel {rel.max()}"


def workload_inputs(name: str):
    w = wl.WORKLOADS[name]
    q, k, v = wl.make_qkv(w)
    seg = wl.make_segment_ids(w)
    return w, q, k, v, seg
