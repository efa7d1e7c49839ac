"""Pins for the oracle's grouped-query attention (CPU only).

The references are torch's library attention with its own grouped-query option
(scaled_dot_product_attention(..., enable_gqa=True) in float64, forward and autograd
backward), central finite differences of a shared key, and a closed form for MQA with
identical query heads.  Planted mistakes (wrong head mapping, no sum over the group) are
shown to fail the library pin.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _rand(B, L, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, L, Hq, D))
    k = rng.standard_normal((B, L, Hkv, D))
    v = rng.standard_normal((B, L, Hkv, D))
    do = rng.standard_normal((B, L, Hq, D))
    return q, k, v, do


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).requires_grad_(True)


def _sdpa_gqa(q, k, v, do, causal):
    tq, tk, tv = _t(q), _t(k), _t(v)
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, enable_gqa=True)
    o.backward(torch.from_numpy(np.ascontiguousarray(do.transpose(0, 2, 1, 3))))
    back = lambda x: x.detach().numpy().transpose(0, 2, 1, 3)   # noqa: E731
    return back(o), back(tq.grad), back(tk.grad), back(tv.grad)


SHAPES = [(1, 37, 4, 2, 8), (2, 129, 6, 1, 16), (1, 64, 3, 3, 8), (1, 200, 8, 2, 32)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,L,Hq,Hkv,D", SHAPES)
def test_gqa_matches_library_attention(causal, B, L, Hq, Hkv, D):
    q, k, v, do = _rand(B, L, Hq, Hkv, D, seed=L + Hq)
    o_ref, dq_ref, dk_ref, dv_ref = _sdpa_gqa(q, k, v, do, causal)
    out, lse = oracle.gqa_fwd(q, k, v, causal)
    assert out.shape == q.shape and lse.shape == (B, Hq, L)
    assert np.max(np.abs(out - o_ref)) < 1e-12
    dq, dk, dv = oracle.gqa_bwd(q, k, v, do, causal)
    assert dk.shape == k.shape and dv.shape == v.shape
    for got, want in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert np.max(np.abs(got - want)) < 1e-11


def test_shared_key_gradient_by_finite_differences():
    q, k, v, do = _rand(1, 9, 4, 2, 3, seed=4)
    _, dk, dv = oracle.gqa_bwd(q, k, v, do, True)
    f = lambda kk, vv: float(np.sum(oracle.gqa_fwd(q, kk, vv, True)[0] * do))   # noqa: E731
    h = 1e-6
    for (c, j, d) in [(0, 0, 0), (3, 1, 2), (8, 1, 1), (5, 0, 1)]:
        kp, km = k.copy(), k.copy()
        kp[0, c, j, d] += h
        km[0, c, j, d] -= h
        assert abs((f(kp, v) - f(km, v)) / (2 * h) - dk[0, c, j, d]) < 1e-7
        vp, vm = v.copy(), v.copy()
        vp[0, c, j, d] += h
        vm[0, c, j, d] -= h
        assert abs((f(k, vp) - f(k, vm)) / (2 * h) - dv[0, c, j, d]) < 1e-7


def test_mqa_with_identical_query_heads():
    """H identical query heads on one KV head: every head's output is the single-head
    output, and the shared dK, dV are H times the single-head gradients."""
    q1, k, v, do1 = _rand(1, 50, 1, 1, 8, seed=5)
    H = 5
    q, do = np.repeat(q1, H, axis=2), np.repeat(do1, H, axis=2)
    o1, _ = oracle.attention_fwd(q1, k, v, True)
    _, dk1, dv1 = oracle.attention_bwd(q1, k, v, do1, True)
    out, _ = oracle.gqa_fwd(q, k, v, True)
    _, dk, dv = oracle.gqa_bwd(q, k, v, do, True)
    assert np.max(np.abs(out - np.repeat(o1, H, axis=2))) < 1e-14
    assert np.max(np.abs(dk - H * dk1)) < 1e-12
    assert np.max(np.abs(dv - H * dv1)) < 1e-12


def test_group_size_rejects_non_divisors():
    assert oracle.group_size(8, 2) == 4
    with pytest.raises(ValueError):
        oracle.group_size(6, 4)
    with pytest.raises(ValueError):
        oracle.group_size(4, 0)


def test_planted_mistakes_fail_the_library_pin():
    q, k, v, do = _rand(1, 40, 4, 2, 8, seed=6)
    o_ref, _, dk_ref, _ = _sdpa_gqa(q, k, v, do, True)
    # query head h on KV head h mod H_kv instead of h // G
    wrong_map = oracle.attention_fwd(q, np.tile(k, (1, 1, 2, 1)), np.tile(v, (1, 1, 2, 1)), True)[0]
    assert np.max(np.abs(wrong_map - o_ref)) > 1e-2
    # dK of the first query head of each group only, no sum over the group
    _, dk_e, _ = oracle.attention_bwd(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2), do,
                                      True)
    assert np.max(np.abs(dk_e[:, :, ::2] - dk_ref)) > 1e-2


@pytest.mark.parametrize("shape", [(1, 37, 4, 2, 8), (1, 64, 3, 1, 16)])
def test_gqa_cols_dkdv_matches_library(shape):
    """The sampled key columns of each shared head against the library's grouped-query
    autograd (the sum over the group included)."""
    q, k, v, do = _rand(*shape, seed=31)
    _, _, gk, gv = _sdpa_gqa(q, k, v, do, True)
    L, Hkv = shape[1], shape[3]
    cols = [0, L // 2, L - 1]
    for hk in range(Hkv):
        dk, dv = oracle.gqa_cols_dkdv(q, k, v, do, 0, hk, cols, causal=True)
        assert np.max(np.abs(dk - gk[0, cols, hk])) < 1e-12
        assert np.max(np.abs(dv - gv[0, cols, hk])) < 1e-12
