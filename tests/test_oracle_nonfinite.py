"""Pins for the oracle on non-finite inputs (CPU only).

labhub "Ring Attention 論文分析", section "限界、失敗事例、そして未解決の問題" (the failure
case "NaN/Inf の発散"), names NaN/Inf arising in the online softmax as a hazard of the
method.  A NaN or an infinity in an input must reach exactly the outputs that the
definition makes depend on it, and no others:

* NaN in one element of q_r: every score of row r is NaN, so out_r, lse_r and dQ_r are NaN;
  row r's terms reach dK_c and dV_c of every key c <= r (causal), so those rows are NaN;
  nothing else changes.
* +inf in feature d of v_c: out_r[d] = +inf for every row r >= c (p[r, c] > 0), nothing else
  of the forward changes; the lse does not involve v.  In the backward dV does not involve v
  (dV_c = sum_r p[r, c] dO_r), so it is unchanged; for rows r >= c, D_r = dO_r . O_r is
  infinite, so dS[r, :] and dQ_r are not finite, and every key is seen by some such row, so
  no dK row is finite; rows r < c never see key c, so their dQ is unchanged.

The poisoned positions are the last row and the first key of a 256-row block, where the
oracle's blocked products hold no masked (zero-probability) term next to the poisoned value.
The forward's NaN pattern is also checked against torch's library attention.
"""

import numpy as np
import torch
import torch.nn.functional as F

import oracle


def _inputs(L=512, H=2, D=16, seed=21):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((1, L, H, D)) for _ in range(4))


def test_nan_in_q_reaches_exactly_its_row_and_the_keys_it_sees():
    q, k, v, do = _inputs()
    r, h = 255, 1                              # last row of the first 256-row block
    qp = q.copy()
    qp[0, r, h, 3] = np.nan
    o, lse = oracle.attention_fwd(qp, k, v, causal=True)
    o0, lse0 = oracle.attention_fwd(q, k, v, causal=True)
    assert np.isnan(o[0, r, h]).all() and np.isnan(lse[0, h, r])
    keep = np.ones(o.shape, bool)
    keep[0, r, h] = False
    assert np.array_equal(o[keep], o0[keep])
    keep_l = np.ones(lse.shape, bool)
    keep_l[0, h, r] = False
    assert np.array_equal(lse[keep_l], lse0[keep_l])
    # the library attention puts its NaNs in the same places
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3)))   # noqa: E731
    ref = F.scaled_dot_product_attention(t(qp), t(k), t(v), is_causal=True).numpy()
    ref = ref.transpose(0, 2, 1, 3)
    assert np.array_equal(np.isnan(ref), np.isnan(o))
    assert np.max(np.abs(ref[keep] - o[keep])) < 1e-12

    dq, dk, dv = oracle.attention_bwd(qp, k, v, do, causal=True)
    dq0, dk0, dv0 = oracle.attention_bwd(q, k, v, do, causal=True)
    assert np.isnan(dq[0, r, h]).all()
    keep = np.ones(dq.shape, bool)
    keep[0, r, h] = False
    assert np.array_equal(dq[keep], dq0[keep])
    for g, g0 in ((dk, dk0), (dv, dv0)):
        assert np.isnan(g[0, :r + 1, h]).all()           # keys c <= r
        keep = np.ones(g.shape, bool)
        keep[0, :r + 1, h] = False
        assert np.array_equal(g[keep], g0[keep])


def test_inf_in_v_reaches_exactly_the_rows_that_see_it():
    q, k, v, do = _inputs()
    c, h, d = 256, 0, 5                        # first key of the second 256-row block
    vp = v.copy()
    vp[0, c, h, d] = np.inf
    o, lse = oracle.attention_fwd(q, k, vp, causal=True)
    o0, lse0 = oracle.attention_fwd(q, k, v, causal=True)
    assert np.array_equal(lse, lse0)
    assert np.isposinf(o[0, c:, h, d]).all()
    keep = np.ones(o.shape, bool)
    keep[0, c:, h, d] = False
    assert np.array_equal(o[keep], o0[keep])

    dq, dk, dv = oracle.attention_bwd(q, k, vp, do, causal=True)
    dq0, dk0, dv0 = oracle.attention_bwd(q, k, v, do, causal=True)
    assert np.array_equal(dv, dv0)
    assert not np.isfinite(dq[0, c:, h]).any()
    assert not np.isfinite(dk[0, :, h]).any()
    keep = np.ones(dq.shape, bool)
    keep[0, c:, h] = False
    assert np.array_equal(dq[keep], dq0[keep])
    keep = np.ones(dk.shape, bool)
    keep[0, :, h] = False
    assert np.array_equal(dk[keep], dk0[keep])


def test_rows_with_no_visible_key_keep_the_guard():
    """Only an empty row takes the guard (p = 0, lse = -inf): a row of -inf scores is not
    a NaN row."""
    p, lse = oracle.attention._softmax_rows(np.array([[-np.inf, -np.inf], [np.nan, 0.0]]))
    assert lse[0] == -np.inf and (p[0] == 0).all()
    assert np.isnan(lse[1]) and np.isnan(p[1]).all()
