"""GPU parity of grouped-query attention (k, v with fewer heads than q) through the C ABI
against the fp64 oracle's gqa_fwd / gqa_bwd.

Tolerances as for plain attention: output max-abs 1e-2 (fp32 output), lse 1e-3,
gradients relative Frobenius 2e-2.  The forward of query head h reads exactly the data the
plain path reads for a KV head repeated G times, so it must match that path bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300.synthetic import make_inputs, to_f64

pytestmark = pytest.mark.gpu

OUT_TOL, LSE_TOL, GRAD_TOL = 1e-2, 1e-3, 2e-2


def _rel(g, r):
    return float(np.linalg.norm(g.float().cpu().numpy() - r) / np.linalg.norm(r))


SWEEP = [
    # B, L, H, H_kv, P, block, layout, causal
    (1, 1024, 4, 2, 4, 128, "striped", True),
    (1, 1024, 4, 1, 4, 128, "contiguous", True),     # MQA
    (2, 1024, 6, 2, 2, 128, "zigzag", True),
    (1, 1536, 8, 2, 4, 128, "striped", True),        # 3 tiles per shard
    (1, 2048, 4, 4, 4, 256, "zigzag", True),         # H_kv = H: plain multi-head
    (1, 1024, 4, 2, 4, 128, "striped", False),
]


@pytest.mark.parametrize("B,L,H,Hkv,P,block,layout,causal", SWEEP)
def test_gqa_parity(B, L, H, Hkv, P, block, layout, causal):
    q, k, v, do = make_inputs(B, L, H, 128, seed=11 * L + H + Hkv, kv_heads=Hkv)
    q64, k64, v64, do64 = to_f64(q, k, v, do)
    o_ref, l_ref = oracle.gqa_fwd(q64, k64, v64, causal)
    dq_r, dk_r, dv_r = oracle.gqa_bwd(q64, k64, v64, do64, causal)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o32, l32 = era.ra_fwd(qd, kd, vd, P, block, layout, causal, out_dtype=torch.float32)
    out, lse = era.ra_fwd(qd, kd, vd, P, block, layout, causal)
    dq, dk, dv = era.ra_bwd(qd, kd, vd, out, lse, dod, P, block, layout, causal)
    torch.cuda.synchronize()
    assert dk.shape == k.shape and dv.shape == v.shape
    assert np.max(np.abs(o32.cpu().numpy() - o_ref)) <= OUT_TOL
    assert np.max(np.abs(l32.cpu().numpy() - l_ref)) <= LSE_TOL
    errs = (_rel(dq, dq_r), _rel(dk, dk_r), _rel(dv, dv_r))
    assert max(errs) <= GRAD_TOL, errs


def test_gqa_forward_equals_repeated_kv_heads_bitwise():
    B, L, H, Hkv, P = 1, 2048, 8, 2, 4
    q, k, v = (t.cuda() for t in make_inputs(B, L, H, 128, seed=3, with_dout=False,
                                             kv_heads=Hkv))
    G = H // Hkv
    ke, ve = k.repeat_interleave(G, dim=2).contiguous(), v.repeat_interleave(G, dim=2).contiguous()
    for layout in ("striped", "zigzag"):
        o1, l1 = era.ra_fwd(q, k, v, P, 128, layout, True)
        o2, l2 = era.ra_fwd(q, ke, ve, P, 128, layout, True)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_gradients_sum_over_the_group():
    B, L, H, Hkv, P = 1, 2048, 8, 2, 4
    q, k, v, do = (t.cuda() for t in make_inputs(B, L, H, 128, seed=4, kv_heads=Hkv))
    G = H // Hkv
    ke, ve = k.repeat_interleave(G, dim=2).contiguous(), v.repeat_interleave(G, dim=2).contiguous()
    out, lse = era.ra_fwd(q, k, v, P, 128, "zigzag", True)
    dq, dk, dv = era.ra_bwd(q, k, v, out, lse, do, P, 128, "zigzag", True)
    dq2, dke, dve = era.ra_bwd(q, ke, ve, out, lse, do, P, 128, "zigzag", True)
    torch.cuda.synchronize()
    dk2 = dke.float().view(B, L, Hkv, G, 128).sum(3)
    dv2 = dve.float().view(B, L, Hkv, G, 128).sum(3)
    assert float((dq.float() - dq2.float()).abs().max()) <= 1e-2
    for got, want in ((dk, dk2), (dv, dv2)):
        assert float((got.float() - want).norm() / want.norm()) <= 1e-2


def test_gqa_rejects_non_dividing_kv_heads():
    q, k, v = (t.cuda() for t in make_inputs(1, 1024, 6, 128, seed=5, with_dout=False,
                                             kv_heads=4))
    with pytest.raises(ValueError):
        era.ra_fwd(q, k, v, 4, 128, "striped", True)


@pytest.mark.parametrize("D,n_split,layout", [(128, 2, "striped"), (64, 1, "zigzag"),
                                              (64, 4, "contiguous")])
def test_gqa_forward_split_and_head_dim_64(D, n_split, layout):
    B, L, H, Hkv, P = 1, 2048, 8, 2, 4
    q, k, v = make_inputs(B, L, H, D, seed=90 + D + n_split, with_dout=False, kv_heads=Hkv)
    q64, k64, v64 = to_f64(q, k, v)
    o_ref, l_ref = oracle.gqa_fwd(q64, k64, v64, True)
    o, l = era.ra_fwd(q.cuda(), k.cuda(), v.cuda(), P, 128, layout, True,
                      out_dtype=torch.float32, n_split=n_split)
    torch.cuda.synchronize()
    assert np.max(np.abs(o.cpu().numpy() - o_ref)) <= OUT_TOL
    assert np.max(np.abs(l.cpu().numpy() - l_ref)) <= LSE_TOL
