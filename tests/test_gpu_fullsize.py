"""GPU parity at the full workload sizes (32k, 262k, 1M tokens), in the launch
configuration the benchmark times.

At 32k tokens the oracle runs whole heads: out, lse, dQ, dK and dV of the first and the
last head are compared with the fp64 oracle element by element.  At 262k and 1M tokens it
computes what it can afford: sampled output rows and lse, sampled dQ rows (O(L*D) each),
and dK, dV of the last 1024 keys of two heads (a key column needs only the rows at or after
it, so the last keys are cheap; in the striped layout they lie in every shard, and they
carry the largest byte offsets).  Identities that hold at any size check every key of every
head besides: the rows of dS sum to zero, so the sum over keys of dK vanishes, and the rows
of P sum to one, so the sum over keys of dV equals the sum over queries of dO.

The oracle's values depend on the workload's inputs, not on the layout, so they are
computed once per workload and head and reused by the layouts.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300.synthetic import WORKLOADS, SEEDS, make_inputs

pytestmark = pytest.mark.gpu

OUT_TOL, LSE_TOL, GRAD_TOL = 1e-2, 1e-3, 2e-2
LAST_KEYS = 1024
WHOLE_HEAD_MAX_L = 32768          # whole-head oracle backward up to this length

_ORACLE = {}                      # (workload, what, head) -> oracle values


def _rows(L, P, layout):
    """Sampled query rows: both ends, shard boundaries and a few interior rows."""
    n = L // P
    picks = {0, 1, L - 1, n - 1, n, L // 2, L // 3 + 7, 5 * L // 7 + 3}
    return sorted(r for r in picks if 0 <= r < L)


def _np(t):
    return t.double().cpu().numpy()


def _rel(got, want):
    return float(np.linalg.norm(got - want) / np.linalg.norm(want))


def _cached(key, fn):
    if key not in _ORACLE:
        _ORACLE[key] = fn()
    return _ORACLE[key]


CASES = [("32k", "striped"), ("262k", "striped"), ("1m", "striped"), ("1m", "contiguous"),
         ("32k", "zigzag"), ("1m", "zigzag"), ("32k-gqa", "zigzag"), ("32k-d64", "zigzag")]


@pytest.mark.parametrize("name,layout", CASES)
def test_fullsize_parity(name, layout):
    w = WORKLOADS[name]
    B, L, H, D, P, blk = (w["batch"], w["seq_len"], w["heads"], w["head_dim"], w["P"],
                          w["block"])
    Hkv = w.get("kv_heads", H)
    G = H // Hkv
    dev = torch.device("cuda:0")
    q, k, v, do = make_inputs(B, L, H, D, SEEDS[name], device=dev, kv_heads=Hkv)
    out, lse = era.ra_fwd(q, k, v, P, blk, layout, True)               # as the bench runs it
    dq, dk, dv = era.ra_bwd(q, k, v, out, lse, do, P, blk, layout, True)
    o32, l32 = era.ra_fwd(q, k, v, P, blk, layout, True, out_dtype=torch.float32)
    torch.cuda.synchronize()

    def head(t, x):                   # one head on the host in float64, [1, L, 1, D]
        return _np(t[0, :, x, :])[None, :, None, :]

    rows = _rows(L, P, layout)
    whole = L <= WHOLE_HEAD_MAX_L and G == 1
    for h in sorted({0, H - 1}):
        qh, doh, kh, vh = head(q, h), head(do, h), head(k, h // G), head(v, h // G)
        ro, rl = _cached((name, "rows", h),
                         lambda: oracle.attention_rows_fwd(qh, kh, vh, 0, 0, rows, causal=True))
        assert np.max(np.abs(_np(o32[0, rows, h, :]) - ro)) <= OUT_TOL
        assert np.max(np.abs(_np(l32[0, h, rows]) - rl)) <= LSE_TOL
        gb = _np(out[0, rows, h, :])
        assert np.all(np.abs(gb - ro) <= OUT_TOL + 2.0 ** -8 * np.abs(ro))
        if whole:
            # the whole head: every output row, and dQ, dK, dV of every token
            wo, wl = _cached((name, "fwd", h),
                             lambda: oracle.attention_fwd(qh, kh, vh, causal=True))
            assert np.max(np.abs(_np(o32[0, :, h, :]) - wo[0, :, 0, :])) <= OUT_TOL
            assert np.max(np.abs(_np(l32[0, h, :]) - wl[0, 0, :])) <= LSE_TOL
            rq, rk, rv = _cached((name, "bwd", h),
                                 lambda: oracle.attention_bwd(qh, kh, vh, doh, causal=True))
            for got, want, nm in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
                e = _rel(_np(got[0, :, h, :]), want[0, :, 0, :])
                assert e <= GRAD_TOL, (nm, h, e)
        else:
            # dQ: a relative Frobenius error over the whole tensor, estimated on a seeded
            # uniform sample of rows (boundary rows would over-weight the few first rows,
            # whose dS = P (dP - D) nearly cancels and so carries the bf16 rounding of O
            # inside D)
            qrows = np.sort(np.random.default_rng(17 + h).choice(L, size=24, replace=False))
            rq = _cached((name, "dq", h), lambda: oracle.attention_rows_dq(
                qh, kh, vh, doh, 0, 0, qrows, causal=True))
            assert _rel(_np(dq[0, qrows, h, :]), rq) <= GRAD_TOL

    if not whole:
        # dK, dV of the last keys of the first and the last key/value head (with grouped
        # query heads: the sum over the group's query heads)
        cols = np.arange(L - LAST_KEYS, L)
        for hk in sorted({0, Hkv - 1}):
            rk, rv = _cached((name, "cols", hk), lambda: oracle.gqa_cols_dkdv(
                _np(q[:, :, hk * G:(hk + 1) * G, :]), head(k, hk), head(v, hk),
                _np(do[:, :, hk * G:(hk + 1) * G, :]), 0, 0, cols, causal=True))
            for got, want, nm in ((dk, rk, "dk"), (dv, rv, "dv")):
                e = _rel(_np(got[0, L - LAST_KEYS:, hk, :]), want)
                assert e <= GRAD_TOL, (nm, hk, e)

    # identities over all keys of every head (float64 sums on the device)
    sk = dk.double().sum(dim=1)
    assert float(sk.norm() / dk.double().norm()) <= GRAD_TOL
    sv = dv.double().sum(dim=1)
    so = do.double().sum(dim=1).view(B, Hkv, G, D).sum(2)      # query heads of each group
    assert float((sv - so).norm() / so.norm()) <= GRAD_TOL
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
