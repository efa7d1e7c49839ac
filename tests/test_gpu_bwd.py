"""GPU parity of the backward path (ra_bwd through the C ABI) against the fp64 oracle.

Tolerance: relative Frobenius error <= 2e-2 for dQ, dK and dV.  The GPU backward takes
the GPU forward's bf16 output and lse, as training would; the oracle's gradients are
the exact ones of the bf16-rounded inputs.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300.synthetic import make_inputs, to_f64

pytestmark = pytest.mark.gpu

GRAD_TOL = 2e-2


def _rel(g, r):
    return float(np.linalg.norm(g.float().cpu().numpy() - r) / np.linalg.norm(r))


def _run(q, k, v, do, P, block, layout, causal):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, lse = era.ra_fwd(qd, kd, vd, P, block, layout, causal)
    dq, dk, dv = era.ra_bwd(qd, kd, vd, out, lse, dod, P, block, layout, causal)
    torch.cuda.synchronize()
    return dq, dk, dv


SWEEP = [
    # B, L, H, P, block, layout, causal
    (1, 1024, 2, 4, 128, "contiguous", True),
    (1, 1024, 2, 4, 128, "striped", True),
    (2, 1024, 3, 2, 128, "striped", True),
    (1, 1024, 2, 8, 128, "contiguous", True),     # one 128-key tile per shard
    (1, 1024, 2, 8, 128, "striped", True),
    (1, 1536, 2, 4, 128, "contiguous", True),     # 3 KV tiles per shard
    (1, 1536, 2, 4, 128, "striped", True),
    (1, 2048, 2, 4, 256, "striped", True),
    (1, 1024, 1, 1, 128, "contiguous", True),     # P = 1
    (1, 1024, 2, 4, 128, "contiguous", False),
    (1, 1024, 2, 4, 128, "striped", False),
    (1, 1024, 2, 4, 128, "zigzag", True),         # one tile per chunk
    (2, 2048, 3, 2, 128, "zigzag", True),
    (1, 1536, 2, 2, 128, "zigzag", True),         # 3 tiles per chunk
    (1, 2048, 2, 4, 256, "zigzag", True),
    (1, 1024, 2, 4, 128, "zigzag", False),
]


@pytest.mark.parametrize("B,L,H,P,block,layout,causal", SWEEP)
def test_bwd_parity_sweep(B, L, H, P, block, layout, causal):
    q, k, v, do = make_inputs(B, L, H, 128, seed=3 * L + H + P)
    q64, k64, v64, do64 = to_f64(q, k, v, do)
    dq_r, dk_r, dv_r = oracle.attention_bwd(q64, k64, v64, do64, causal)
    dq, dk, dv = _run(q, k, v, do, P, block, layout, causal)
    errs = (_rel(dq, dq_r), _rel(dk, dk_r), _rel(dv, dv_r))
    assert max(errs) <= GRAD_TOL, errs


def test_bwd_invariants_and_determinism():
    q, k, v, do = make_inputs(1, 4096, 4, 128, seed=21)
    dq, dk, dv = _run(q, k, v, do, 8, 128, "striped", True)
    dkf, dvf = dk.float().cpu(), dv.float().cpu()
    # rows of dS sum to zero -> sum over keys of dK vanishes (relative to its size)
    assert float(dkf.sum(1).norm() / dkf.norm()) < 2e-2
    # rows of P sum to one -> sum over keys of dV equals sum over queries of dO
    ref = do.float().sum(1)
    assert float((dvf.sum(1) - ref).norm() / ref.norm()) < 2e-2
    # dK and dV are written by one CTA each: bitwise deterministic
    dq2, dk2, dv2 = _run(q, k, v, do, 8, 128, "striped", True)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert float((dq.float() - dq2.float()).abs().max()) <= 1e-2


def test_bwd_layouts_agree():
    q, k, v, do = make_inputs(1, 4096, 2, 128, seed=22)
    a = _run(q, k, v, do, 8, 128, "contiguous", True)
    b = _run(q, k, v, do, 8, 128, "striped", True)
    z = _run(q, k, v, do, 8, 128, "zigzag", True)
    for x, y, w in zip(a, b, z):
        assert float((x.float() - y.float()).norm() / y.float().norm()) <= GRAD_TOL
        assert float((w.float() - y.float()).norm() / y.float().norm()) <= GRAD_TOL


@pytest.mark.parametrize("B,L,H,Hkv,P,block,layout,causal", [
    (1, 2048, 2, 2, 4, 128, "striped", True),
    (2, 1536, 3, 3, 4, 128, "contiguous", True),    # 3 KV tiles per shard, batch 2
    (1, 2048, 4, 2, 4, 256, "zigzag", True),        # grouped-query, 2:1
    (1, 1024, 2, 1, 1, 128, "contiguous", True),    # P = 1, one KV head
    (1, 1024, 2, 2, 4, 128, "striped", False),
])
def test_bwd_head_dim_64(B, L, H, Hkv, P, block, layout, causal):
    # head_dim 64: the kernel keeps K 128 features wide (the upper half zero) so that
    # dQ^T = K^T dS^T is still an M = 128 product; only its first 64 rows are drained
    q, k, v, do = make_inputs(B, L, H, 64, seed=640 + L + H, kv_heads=Hkv)
    q64, k64, v64, do64 = to_f64(q, k, v, do)
    dq_r, dk_r, dv_r = oracle.gqa_bwd(q64, k64, v64, do64, causal)
    dq, dk, dv = _run(q, k, v, do, P, block, layout, causal)
    errs = (_rel(dq, dq_r), _rel(dk, dk_r), _rel(dv, dv_r))
    assert max(errs) <= GRAD_TOL, errs
