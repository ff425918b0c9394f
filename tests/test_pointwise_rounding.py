"""The pointwise path's relative tolerance, derived from its roundings.

The HSTU forward (hstu_ops ``_pointwise_splash_attention_fwd_kernel_impl``)
computes the activated scores in f32 and multiplies them by f32 values.  The
CUDA path computes q.k with an f32 accumulator, p = x*sigmoid(x)/Sq in f32,
keeps p as two bf16 numbers (hi = bf16(p), lo = bf16(p - hi)) for the two
P.V products, accumulates O in f32 and rounds O to bf16.  This test applies
exactly those roundings to the inputs on the CPU (no CUDA path involved) and
checks that the result stays inside the 2e-3 relative mean gate the GPU
tests use, with a margin -- and that a single bf16 rounding of p would not.
The oracle is the fp64 definition.
"""

import math

import numpy as np
import torch

import oracle
from block_sparse_masked_build_gb300 import workloads as wl
from gpu_helpers import PW_MEAN_REL


def _bf16(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def _emulate(q, k, v, scale, split):
    """Pointwise attention with the CUDA path's roundings (causal, one
    head): f32 scores and activation, p as bf16 (hi [+ lo]), bf16 out."""
    qf = q[0, 0].float().numpy()
    kf = k[0, 0].float().numpy()
    vf = v[0, 0].double().numpy()
    S = qf.shape[0]
    s = (qf @ kf.T).astype(np.float32)                      # f32 accumulate
    x = (s * np.float32(scale)).astype(np.float32)
    sig = (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)
    p = (x * sig * np.float32(1.0 / S)).astype(np.float32)
    p = np.where(np.tril(np.ones((S, S), dtype=bool)), p, np.float32(0.0))
    hi = _bf16(p)
    pe = hi + (_bf16(p - hi.astype(np.float32)) if split else 0.0)
    return _bf16(pe @ vf)                                   # bf16 out


def _rel_mean(got, ref):
    return float(np.abs(got - ref).mean() / np.abs(ref).mean())


def test_split_p_meets_relative_gate_single_bf16_does_not():
    for scale_kind in ("inv_sqrt_d", "inv_s"):
        w = wl.WORKLOADS["cfg4p_hstu_s4096_d128"].with_(S=2048)
        if scale_kind == "inv_s":
            w = w.with_(scale=1.0 / w.S)
        q, k, v = wl.make_qkv(w, B=1, H=1)
        ref = oracle.pointwise_attention(q, k, v, wl.MASK_CAUSAL, 0, None,
                                         None, w.scale)[0, 0]
        split = _rel_mean(_emulate(q, k, v, w.scale, True), ref)
        single = _rel_mean(_emulate(q, k, v, w.scale, False), ref)
        assert split <= 0.8 * PW_MEAN_REL, (scale_kind, split)
        assert single > PW_MEAN_REL, (scale_kind, single)
        assert math.isfinite(split) and split > 0
