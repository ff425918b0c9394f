"""Pins of the oracle's backward (gradients of both score paths).

The analytic gradients are checked against central finite differences of
the forward oracle itself -- an independent route: only the forward
definitions and the loss sum(do * out) are shared -- on tiny float64 shapes
under every mask kind, plus invariants of each score path.
"""

import numpy as np
import pytest

import oracle
from oracle import (MASK_BAND, MASK_CAUSAL, MASK_DENSE, MASK_LOCAL,
                    MASK_SEGMENT)

S, D = 11, 4


def _inputs(seed, H=2, B=2, Skv=S):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, S, D))
    k = rng.standard_normal((B, H, Skv, D))
    v = rng.standard_normal((B, H, Skv, D))
    do = rng.standard_normal((B, H, S, D))
    return q, k, v, do


def _masks():
    rng = np.random.default_rng(5)
    seg = np.array([[0] * 4 + [1] * 5 + [2] * 2, [0] * 7 + [1] * 4],
                   dtype=np.int32)
    dense = rng.random((S, S)) < 0.6
    return [
        (0, 0, None, None), (MASK_CAUSAL, 0, None, None),
        (MASK_CAUSAL | MASK_LOCAL, 3, None, None),
        (MASK_LOCAL | MASK_BAND, 2, None, None),
        (MASK_CAUSAL | MASK_SEGMENT, 0, seg, None),
        (MASK_DENSE, 0, None, dense),
    ]


def _loss(fwd, q, k, v, do, flags, window, seg, dense, scale):
    out = fwd(q, k, v, flags, window, seg, seg, scale, dense=dense)
    out = out[0] if isinstance(out, tuple) else out
    return float((do * out).sum())


def _finite_diff(fwd, x_index, q, k, v, do, flags, window, seg, dense, scale,
                 h=1e-6):
    xs = [q, k, v]
    x = xs[x_index]
    g = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        old = x[idx]
        x[idx] = old + h
        lp = _loss(fwd, *xs, do, flags, window, seg, dense, scale)
        x[idx] = old - h
        lm = _loss(fwd, *xs, do, flags, window, seg, dense, scale)
        x[idx] = old
        g[idx] = (lp - lm) / (2 * h)
    return g


@pytest.mark.parametrize("m", range(6))
@pytest.mark.parametrize("path", ["softmax", "pointwise"])
def test_gradients_match_finite_differences(m, path):
    flags, window, seg, dense = _masks()[m]
    q, k, v, do = _inputs(40 + m)
    scale = 0.7
    if path == "softmax":
        fwd, bwd = oracle.softmax_attention, oracle.softmax_attention_bwd
    else:
        fwd, bwd = oracle.pointwise_attention, oracle.pointwise_attention_bwd
    grads = bwd(q, k, v, do, flags, window, seg, seg, scale, dense=dense)
    for i, g in enumerate(grads):
        fd = _finite_diff(fwd, i, q, k, v, do, flags, window, seg, dense,
                          scale)
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-8,
                                   err_msg=f"{path} d{'qkv'[i]} mask {m}")


def test_softmax_key_gradients_sum_to_zero():
    # softmax is unchanged when every visible key moves by the same vector,
    # so the key gradients of each (b, h) add up to zero
    q, k, v, do = _inputs(7)
    _, dk, _ = oracle.softmax_attention_bwd(q, k, v, do, MASK_CAUSAL, 0, None,
                                            None, 0.5)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)


def test_pointwise_dv_does_not_depend_on_v_and_dq_is_linear_in_do():
    q, k, v, do = _inputs(8)
    a = oracle.pointwise_attention_bwd(q, k, v, do, MASK_CAUSAL, 0, None,
                                       None, 0.5)
    b = oracle.pointwise_attention_bwd(q, k, 3 * v + 1, do, MASK_CAUSAL, 0,
                                       None, None, 0.5)
    np.testing.assert_allclose(a[2], b[2], rtol=0, atol=1e-12)
    c = oracle.pointwise_attention_bwd(q, k, v, 2 * do, MASK_CAUSAL, 0, None,
                                       None, 0.5)
    np.testing.assert_allclose(c[0], 2 * a[0], rtol=1e-12, atol=1e-12)


def test_fully_masked_rows_and_hidden_keys_get_no_gradient():
    # an arbitrary mask that hides row 3 entirely and key 5 from every row
    q, k, v, do = _inputs(9)
    dense = np.ones((S, S), dtype=bool)
    dense[3, :] = False
    dense[:, 5] = False
    for bwd in (oracle.softmax_attention_bwd, oracle.pointwise_attention_bwd):
        dq, dk, dv = bwd(q, k, v, do, MASK_DENSE, 0, None, None, 0.5,
                         dense=dense)
        assert not dq[:, :, 3].any()
        assert not dk[:, :, 5].any() and not dv[:, :, 5].any()
