"""Plain fp64 definitions of the block-sparse masked attention forward pass.

Test infrastructure only (see the package docstring).  All floating point is
numpy float64; bfloat16 inputs are upcast exactly.  No blocking, fusion or
reordering is done beyond what each cited definition states; the only
library primitives used are matrix products, ``exp``/``log`` and
``logaddexp``.

Readings taken where the pages leave a point open:

* Elements outside [0, Sq) x [0, Skv) (a ragged last block) are invisible.
* The local window with causal means visible iff 0 <= q - k < window.
* Segment ids mask an element iff q_seg != kv_seg (hstu_ops ``_apply_mask``,
  the ``q_ids == kv_ids`` term).
* A fully masked softmax row gives out = 0 and lse = -inf.
* The pointwise output is the SUM over all visible keys (the hstu_ops
  forward assigns ``o_ref[:] = o_curr`` per step as printed, but its
  backward differentiates the sum, and the splash notes section 14 state that
  KV tiles add up), with the fixed ``1/seq_len`` factor where seq_len is the
  query length.
* ``data_next[i, j]`` is the smallest nonzero block index >= j in row i; when
  none is left, the largest nonzero index < j; 0 for an empty row (section 21
  of the splash notes: empty steps point at a nonzero block, e.g. with valid
  flags 1 0 0 1 0 1, steps 1 and 2 point at block 3).
"""

from __future__ import annotations

import numpy as np

MASK_CAUSAL = 1
MASK_LOCAL = 2
MASK_SEGMENT = 4
MASK_BAND = 8
MASK_DENSE = 16


def _f64(x) -> np.ndarray:
    """Exact upcast of a torch (bf16/f32) tensor or array to numpy float64."""
    try:
        import torch  # local: the oracle itself does not need torch otherwise

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def visible(flags, window, qi, ki, Sq, Skv, q_seg=None, kv_seg=None,
            dense=None):
    """Per-element visibility (broadcasts qi against ki).

    Causal: k <= q (CausalMask, offset 0; hstu_ops ``pointwise_splash_attention``
    MaskType.CAUSAL).  Local: q - k < window (the local-window workload's
    "(q-k) < 4096").  Band (with local): also k - q < window, the symmetric
    window of hstu_ops ``LocalMask((w, w))``.  Segment: q_seg[q] == kv_seg[k]
    (hstu_ops ``_apply_mask``).  Dense: an arbitrary boolean [Sq, Skv] mask,
    dense[q, k] (hstu_ops ``NumpyMask``).  Full mask: every in-range element
    (MaskType.FULL).
    """
    qi = np.asarray(qi)
    ki = np.asarray(ki)
    vis = (qi < Sq) & (ki < Skv) & (qi >= 0) & (ki >= 0)
    if flags & MASK_CAUSAL:
        vis = vis & (ki <= qi)
    if flags & MASK_LOCAL:
        vis = vis & ((qi - ki) < window)
    if flags & MASK_BAND:
        vis = vis & ((ki - qi) < window)
    if flags & MASK_SEGMENT:
        qs = np.asarray(q_seg)[np.clip(qi, 0, Sq - 1)]
        ks = np.asarray(kv_seg)[np.clip(ki, 0, Skv - 1)]
        vis = vis & (qs == ks)
    if flags & MASK_DENSE:
        dm = np.asarray(dense, dtype=bool)
        vis = vis & dm[np.clip(qi, 0, Sq - 1), np.clip(ki, 0, Skv - 1)]
    return vis


def visibility_matrix(flags, window, Sq, Skv, q_seg=None, kv_seg=None,
                      rows=None, dense=None):
    """Boolean [len(rows), Skv] visibility for one batch row's segment ids."""
    qi = np.arange(Sq) if rows is None else np.asarray(rows)
    ki = np.arange(Skv)
    return visible(flags, window, qi[:, None], ki[None, :], Sq, Skv,
                   q_seg, kv_seg, dense)


def mask_info(flags, window, q_seg, kv_seg, B, Sq, Skv, bq, bkv, dense=None):
    """Brute-force mask-info by an exact per-element scan of every block.

    Class encoding from hstu_ops ``_next_nonzero``: 0 = empty (block not
    run), 1 = partial (the element mask is applied), 2 = full (no mask).
    Block (i, j) covers rows [i*bq, (i+1)*bq) and columns [j*bkv, (j+1)*bkv);
    elements past Sq or Skv count as invisible.  One table per batch row when
    segment ids are used, else one table shared by every batch row and head
    (the same mask for every head, as ``MultiHeadMask`` is built in
    ``pointwise_splash_attention``).

    Returns a dict of numpy arrays:
      block_mask int8 [B', nq, nk], data_next int32 [B', nq, nk],
      row_ptr int32 [B'*nq + 1], kv_idx int32 [nnz], kv_cls int8 [nnz].
    """
    nq = -(-Sq // bq)
    nk = -(-Skv // bkv)
    Bp = B if flags & MASK_SEGMENT else 1
    block_mask = np.zeros((Bp, nq, nk), dtype=np.int8)
    data_next = np.zeros((Bp, nq, nk), dtype=np.int32)
    cols = np.arange(nk * bkv)
    kv_idx, kv_cls = [], []
    row_ptr = [0]
    for b in range(Bp):
        qs = None if q_seg is None else np.asarray(q_seg)[b]
        ks = None if kv_seg is None else np.asarray(kv_seg)[b]
        for i in range(nq):
            rows = np.arange(i * bq, (i + 1) * bq)
            vis = visible(flags, window, rows[:, None], cols[None, :], Sq, Skv,
                          qs, ks, dense)
            cnt = vis.reshape(bq, nk, bkv).sum(axis=(0, 2))
            cls = np.where(cnt == 0, 0, np.where(cnt == bq * bkv, 2, 1))
            block_mask[b, i] = cls
            nz = np.flatnonzero(cls > 0)
            if len(nz):
                pos = np.searchsorted(nz, np.arange(nk), side="left")
                nxt = np.where(pos < len(nz), nz[np.minimum(pos, len(nz) - 1)],
                               nz[-1])
                data_next[b, i] = nxt
            kv_idx.extend(nz.tolist())
            kv_cls.extend(cls[nz].tolist())
            row_ptr.append(len(kv_idx))
    return {
        "block_mask": block_mask,
        "data_next": data_next,
        "row_ptr": np.asarray(row_ptr, dtype=np.int32),
        "kv_idx": np.asarray(kv_idx, dtype=np.int32),
        "kv_cls": np.asarray(kv_cls, dtype=np.int8),
        "nq": nq,
        "nk": nk,
        "Bp": Bp,
    }


def visible_pair_count(flags, window, q_seg, kv_seg, B, Sq, Skv, slab=1024,
                       dense=None):
    """Number of visible (q, k) pairs summed over batch rows (per head)."""
    total = 0
    for b in range(B):
        qs = None if q_seg is None else np.asarray(q_seg)[b]
        ks = None if kv_seg is None else np.asarray(kv_seg)[b]
        for r0 in range(0, Sq, slab):
            rows = np.arange(r0, min(Sq, r0 + slab))
            total += int(visibility_matrix(flags, window, Sq, Skv, qs, ks,
                                           rows, dense).sum())
    return total


def unmasked_flops(flags, window, q_seg, kv_seg, B, H, Sq, Skv, D):
    """4*D flops per visible (q, k) pair: 2*D for q.k and 2*D for p*v."""
    return 4 * D * H * visible_pair_count(flags, window, q_seg, kv_seg, B,
                                          Sq, Skv)


def _row_groups(B, H, Sq, rows):
    if rows is None:
        for b in range(B):
            for h in range(H):
                yield b, h, np.arange(Sq)
        return
    rows = list(rows)
    by_bh: dict[tuple[int, int], list[int]] = {}
    for (b, h, q) in rows:
        by_bh.setdefault((b, h), []).append(q)
    for (b, h), qs in by_bh.items():
        yield b, h, np.asarray(qs)


def softmax_attention(q, k, v, flags, window, q_seg, kv_seg, scale,
                      rows=None, slab=512, dense=None):
    """Masked softmax attention, materialised, two passes per row.

    Splash notes section 12 (naive attention: scores = Q K^T, mask, row max,
    exp, row sum, normalise, times V) and section 15:
      Out = sum_t e^{a_t - M} v_t / sum_t e^{a_t - M},  M = max_t a_t,
    with a_t = scale * q . k_t over the visible keys only.  lse = M + ln L
    (natural log of sum_t e^{a_t} over visible t).

    ``rows=None`` computes every row: returns out [B,H,Sq,D], lse [B,H,Sq].
    Otherwise ``rows`` is a list of distinct (b, h, q) and the result is
    out [n, D], lse [n] in the order of ``rows``.
    """
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    B, H, Sq, D = qf.shape
    Skv = kf.shape[2]
    if rows is None:
        out = np.zeros((B, H, Sq, D))
        lse = np.full((B, H, Sq), -np.inf)
    else:
        order = _order(rows)
        out = np.zeros((len(order), D))
        lse = np.full((len(order),), -np.inf)
    for b, h, qrows in _row_groups(B, H, Sq, rows):
        qs = None if q_seg is None else np.asarray(q_seg)[b]
        ks = None if kv_seg is None else np.asarray(kv_seg)[b]
        for s0 in range(0, len(qrows), slab):
            rr = qrows[s0:s0 + slab]
            a = scale * (qf[b, h, rr] @ kf[b, h].T)          # [r, Skv]
            vis = visibility_matrix(flags, window, Sq, Skv, qs, ks, rr, dense)
            a = np.where(vis, a, -np.inf)
            M = a.max(axis=1)                                 # [r]
            any_vis = vis.any(axis=1)
            Msafe = np.where(any_vis, M, 0.0)
            e = np.where(vis, np.exp(a - Msafe[:, None]), 0.0)
            L = e.sum(axis=1)
            O = e @ vf[b, h]                                  # [r, D]
            o = np.where(any_vis[:, None], O / np.where(any_vis, L, 1.0)[:, None],
                         0.0)
            l_ = np.where(any_vis, Msafe + np.log(np.where(any_vis, L, 1.0)),
                          -np.inf)
            if rows is None:
                out[b, h, rr] = o
                lse[b, h, rr] = l_
            else:
                for n, qq in enumerate(rr):
                    idx = order[(b, h, int(qq))]
                    out[idx] = o[n]
                    lse[idx] = l_[n]
    return out, lse


def softmax_attention_online(q, k, v, flags, window, q_seg, kv_seg, scale,
                             block_kv, b=0, h=0, dense=None):
    """Online softmax over KV blocks of ``block_kv`` keys for one (b, h).

    Splash notes section 15.1-15.3: per block B, m_new = max(m, max_B a);
    alpha = e^{m - m_new}; l = alpha*l + sum_B e^{a - m_new};
    o = alpha*o + sum_B e^{a - m_new} v; at the end Out = o / l.
    Used only to pin the two-pass definition (the result must not depend on
    the block size).  Returns out [Sq, D], lse [Sq].
    """
    qf, kf, vf = _f64(q)[b, h], _f64(k)[b, h], _f64(v)[b, h]
    Sq, D = qf.shape
    Skv = kf.shape[0]
    qs = None if q_seg is None else np.asarray(q_seg)[b]
    ks = None if kv_seg is None else np.asarray(kv_seg)[b]
    m = np.full(Sq, -np.inf)
    l = np.zeros(Sq)
    o = np.zeros((Sq, D))
    rows = np.arange(Sq)
    for j0 in range(0, Skv, block_kv):
        cols = np.arange(j0, min(Skv, j0 + block_kv))
        a = scale * (qf @ kf[cols].T)
        vis = visible(flags, window, rows[:, None], cols[None, :], Sq, Skv,
                      qs, ks, dense)
        a = np.where(vis, a, -np.inf)
        m_new = np.maximum(m, a.max(axis=1))
        alive = np.isfinite(m_new)
        m_safe = np.where(alive, m_new, 0.0)
        alpha = np.where(np.isfinite(m), np.exp(m - m_safe), 0.0)
        p = np.where(vis, np.exp(a - m_safe[:, None]), 0.0)
        l = alpha * l + p.sum(axis=1)
        o = alpha[:, None] * o + p @ vf[cols]
        m = m_new
    nz = l > 0
    out = np.where(nz[:, None], o / np.where(nz, l, 1.0)[:, None], 0.0)
    lse = np.where(nz, m + np.log(np.where(nz, l, 1.0)), -np.inf)
    return out, lse


def _silu(x):
    """x * sigmoid(x) in fp64, sigmoid(x) = exp(-log(1 + e^{-x}))."""
    return x * np.exp(-np.logaddexp(0.0, -x))


def pointwise_attention(q, k, v, flags, window, q_seg, kv_seg, scale,
                        rows=None, slab=512, dense=None):
    """Pointwise (HSTU) attention, materialised.

    hstu_ops ``_pointwise_splash_attention_fwd_kernel_impl``: qk = q . k (f32
    accumulate), qk *= scale, qk = qk * logistic(qk) * (1 / seq_len) with
    seq_len the query length, masked elements set to 0 (``_apply_mask``:
    ``where(mask, qk, 0)``), out = sum over keys of qk * v.  No max, no sum,
    no normalisation, no logsumexp.
    """
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    B, H, Sq, D = qf.shape
    Skv = kf.shape[2]
    if rows is None:
        out = np.zeros((B, H, Sq, D))
    else:
        order = _order(rows)
        out = np.zeros((len(order), D))
    for b, h, qrows in _row_groups(B, H, Sq, rows):
        qs = None if q_seg is None else np.asarray(q_seg)[b]
        ks = None if kv_seg is None else np.asarray(kv_seg)[b]
        for s0 in range(0, len(qrows), slab):
            rr = qrows[s0:s0 + slab]
            x = scale * (qf[b, h, rr] @ kf[b, h].T)
            p = _silu(x) * (1.0 / Sq)
            vis = visibility_matrix(flags, window, Sq, Skv, qs, ks, rr, dense)
            p = np.where(vis, p, 0.0)
            o = p @ vf[b, h]
            if rows is None:
                out[b, h, rr] = o
            else:
                for n, qq in enumerate(rr):
                    out[order[(b, h, int(qq))]] = o[n]
    return out


def _order(rows):
    """Position of each (b, h, q) in the caller's ``rows`` list."""
    return {(int(b), int(h), int(q)): n for n, (b, h, q) in enumerate(rows)}


def _bwd_inputs(q, k, v, do):
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    if kf.shape[1] != qf.shape[1]:
        raise ValueError("the backward oracle takes as many K/V heads as "
                         "query heads")
    return qf, kf, vf, dof


def softmax_attention_bwd(q, k, v, do, flags, window, q_seg, kv_seg, scale,
                          dense=None):
    """Gradients (dq, dk, dv) of sum(do * out) for the softmax path.

    The forward of ``softmax_attention``, differentiated as written: with
    s = scale * q k^T over the visible keys, P = softmax(s) per row and
    out = P v,
      dv = P^T do,  dP = do v^T,  D_q = sum_d do[q, d] out[q, d],
      ds = P * (dP - D_q),  dq = scale * ds k,  dk = scale * ds^T q.
    A row that sees no key has P = 0 and adds nothing.  Shapes as the
    forward ([B, H, S, D]); returns float64 arrays.
    """
    qf, kf, vf, dof = _bwd_inputs(q, k, v, do)
    B, H, Sq, D = qf.shape
    Skv = kf.shape[2]
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    for b in range(B):
        qs = None if q_seg is None else np.asarray(q_seg)[b]
        ks = None if kv_seg is None else np.asarray(kv_seg)[b]
        vis = visibility_matrix(flags, window, Sq, Skv, qs, ks, None, dense)
        any_vis = vis.any(axis=1)
        for h in range(H):
            a = np.where(vis, scale * (qf[b, h] @ kf[b, h].T), -np.inf)
            M = np.where(any_vis, a.max(axis=1), 0.0)
            e = np.where(vis, np.exp(a - M[:, None]), 0.0)
            L = e.sum(axis=1)
            P = e / np.where(any_vis, L, 1.0)[:, None]
            out = P @ vf[b, h]
            dv[b, h] = P.T @ dof[b, h]
            dP = dof[b, h] @ vf[b, h].T
            Dq = (dof[b, h] * out).sum(axis=1)
            ds = P * (dP - Dq[:, None])
            dq[b, h] = scale * (ds @ kf[b, h])
            dk[b, h] = scale * (ds.T @ qf[b, h])
    return dq, dk, dv


def pointwise_attention_bwd(q, k, v, do, flags, window, q_seg, kv_seg, scale,
                            dense=None):
    """Gradients (dq, dk, dv) of sum(do * out) for the pointwise path.

    hstu_ops ``_pointwise_splash_attention_bwd_kernel_impl``: with
    x = scale * q k^T, sig = logistic(x) (0 where masked) and
    p = x * sig / Sq,
      dv = p^T do,  dp = (do v^T) * sig * (1 + x (1 - sig)) / Sq,
      dq = scale * dp k,  dk = scale * dp^T q,
    each summed over every visible key (the kernel accumulates dk and dv over
    query blocks and dq over key blocks).  Sq is the query length.
    """
    qf, kf, vf, dof = _bwd_inputs(q, k, v, do)
    B, H, Sq, D = qf.shape
    Skv = kf.shape[2]
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    for b in range(B):
        qs = None if q_seg is None else np.asarray(q_seg)[b]
        ks = None if kv_seg is None else np.asarray(kv_seg)[b]
        vis = visibility_matrix(flags, window, Sq, Skv, qs, ks, None, dense)
        for h in range(H):
            x = scale * (qf[b, h] @ kf[b, h].T)
            sig = np.where(vis, np.exp(-np.logaddexp(0.0, -x)), 0.0)
            p = x * sig / Sq
            dv[b, h] = p.T @ dof[b, h]
            dp = (dof[b, h] @ vf[b, h].T) * sig * (1.0 + x * (1.0 - sig)) / Sq
            dq[b, h] = scale * (dp @ kf[b, h])
            dk[b, h] = scale * (dp.T @ qf[b, h])
    return dq, dk, dv

