"""The backward's tolerance, derived from its roundings.

The CUDA backward computes s = scale * q.k with an f32 accumulator, P (and
for the softmax path D_q from the bf16 forward output), rounds P and dS to
bf16 for the products -- as hstu_ops' backward casts p to the input type --
accumulates dQ, dK, dV in f32 and rounds them to bf16.  This test applies
exactly those roundings on the CPU (no CUDA path involved), compares with
the fp64 backward oracle, and checks that the relative errors sit inside
the gates the GPU tests use (mean error <= 4e-3 * mean |ref|, max error
<= 2e-2 * max |ref|) with a margin: two bf16 roundings give ~2.3e-3.
"""

import numpy as np
import torch

import oracle
from gpu_helpers import BWD_MAX_REL, BWD_MEAN_REL


def _bf16(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def _emulate(q, k, v, do, score, flags, scale):
    qf, kf, vf, dof = (t[0, 0].double().numpy() for t in (q, k, v, do))
    S = qf.shape[0]
    vis = oracle.visibility_matrix(flags, 0, S, S)
    x = ((qf @ kf.T).astype(np.float32) * np.float32(scale)).astype(np.float64)
    dp = (dof @ vf.T).astype(np.float32).astype(np.float64)
    if score == 0:
        out, lse = oracle.softmax_attention(q, k, v, flags, 0, None, None,
                                            scale)
        p = np.where(vis, np.exp(x - lse[0, 0][:, None]), 0.0)
        dq_ = (dof * _bf16(out[0, 0])).sum(axis=1)
        ds = p * (dp - dq_[:, None])
    else:
        sig = 1.0 / (1.0 + np.exp(-x))
        p = np.where(vis, x * sig / S, 0.0)
        ds = np.where(vis, dp * sig * (1.0 + x * (1.0 - sig)) / S, 0.0)
    pb, dsb = _bf16(p), _bf16(ds)
    return (_bf16(scale * dsb @ kf), _bf16(scale * dsb.T @ qf),
            _bf16(pb.T @ dof))


def test_backward_roundings_meet_the_gates():
    for score, sigma, seed in ((0, 1.0, 3), (1, 0.5, 4)):
        g = torch.Generator().manual_seed(seed)
        S, D = 384, 128
        q, k, v, do = ((torch.randn(1, 1, S, D, generator=g) * sigma)
                       .to(torch.bfloat16) for _ in range(4))
        scale = 1.0 / np.sqrt(D)
        bwd = oracle.softmax_attention_bwd if score == 0 else \
            oracle.pointwise_attention_bwd
        ref = bwd(q, k, v, do, oracle.MASK_CAUSAL, 0, None, None, scale)
        got = _emulate(q, k, v, do, score, oracle.MASK_CAUSAL, scale)
        for name, gv, rv in zip(("dq", "dk", "dv"), got, ref):
            r = rv[0, 0]
            err = np.abs(gv - r)
            mean_rel = err.mean() / np.abs(r).mean()
            max_rel = err.max() / np.abs(r).max()
            assert 1e-3 < mean_rel <= 0.7 * BWD_MEAN_REL, (score, name, mean_rel)
            assert max_rel <= 0.5 * BWD_MAX_REL, (score, name, max_rel)
