"""Pins for the fp64 oracle's exact attention (CPU only).

Each test checks the oracle against something other than itself: a library softmax
attention (torch's scaled_dot_product_attention on CPU in float64), a pure-Python
triple loop, closed forms, invariants, or central finite differences.  The last tests
plant mistakes in the oracle and check that the pins catch them.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attention as oatt


def _rand(B, L, H, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return tuple(scale * rng.standard_normal((B, L, H, D)) for _ in range(4))


def _sdpa(q, k, v, causal):
    """torch's library attention in float64 on the CPU, [B,L,H,D] in and out."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3)))
                  for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
    return o.numpy().transpose(0, 2, 1, 3)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 37, 2, 8), (2, 300, 1, 16), (1, 513, 3, 64)])
def test_fwd_matches_library_attention(causal, shape):
    q, k, v, _ = _rand(*shape, seed=1)
    out, _ = oracle.attention_fwd(q, k, v, causal)
    ref = _sdpa(q, k, v, causal)
    assert np.max(np.abs(out - ref)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_matches_brute_force(causal):
    q, k, v, _ = _rand(1, 19, 2, 5, seed=2)
    out, lse = oracle.attention_fwd(q, k, v, causal, scale=0.37)
    bo, bl = oracle.brute_force_fwd(q, k, v, causal, scale=0.37)
    assert np.max(np.abs(out - bo)) < 1e-13
    assert np.max(np.abs(lse - bl)) < 1e-13


def test_lse_is_natural_log_of_row_sum():
    # lse against a direct log-sum-exp of explicitly built scores (scipy, library)
    from scipy.special import logsumexp
    q, k, v, _ = _rand(1, 40, 1, 8, seed=3)
    _, lse = oracle.attention_fwd(q, k, v, causal=True)
    s = (q[0, :, 0, :] @ k[0, :, 0, :].T) / math.sqrt(8)
    for r in range(40):
        assert abs(lse[0, 0, r] - logsumexp(s[r, :r + 1])) < 1e-13


def test_single_key_gives_v_and_score():
    q, k, v, _ = _rand(1, 1, 1, 8, seed=4)
    out, lse = oracle.attention_fwd(q, k, v, causal=False)
    assert np.array_equal(out, v)
    assert abs(lse[0, 0, 0] - float(q[0, 0, 0] @ k[0, 0, 0]) / math.sqrt(8)) < 1e-15


def test_first_causal_token():
    q, k, v, _ = _rand(2, 64, 3, 16, seed=5)
    out, lse = oracle.attention_fwd(q, k, v, causal=True)
    assert np.array_equal(out[:, 0], v[:, 0])
    s00 = np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]) / 4.0
    assert np.max(np.abs(lse[:, :, 0] - s00)) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    # with V = one-hot rows (v_c = e_c), out_r is exactly the probability row p_r
    L = 24
    q, k, _, _ = _rand(1, L, 1, L, seed=6)
    v = np.eye(L)[None, :, None, :]
    out, _ = oracle.attention_fwd(q, k, v, causal)
    p = out[0, :, 0, :]
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-14
    assert np.all(p >= 0)
    if causal:
        assert np.all(np.triu(p, 1) == 0)


def test_constant_v_gives_constant_out_and_zero_dq_dk():
    q, k, _, dout = _rand(1, 50, 2, 8, seed=7)
    v = np.broadcast_to(np.linspace(-2, 3, 8), q.shape).copy()
    for causal in (False, True):
        out, _ = oracle.attention_fwd(q, k, v, causal)
        assert np.max(np.abs(out - v)) < 1e-14
        dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal)
        assert np.max(np.abs(dq)) < 1e-13 and np.max(np.abs(dk)) < 1e-13


def test_key_shift_invariance():
    q, k, v, _ = _rand(1, 33, 2, 8, seed=8)
    w = np.random.default_rng(9).standard_normal(8)
    for causal in (False, True):
        o1, l1 = oracle.attention_fwd(q, k, v, causal)
        o2, l2 = oracle.attention_fwd(q, k + w, v, causal)
        shift = np.einsum("blhd,d->bhl", q, w) / math.sqrt(8)
        assert np.max(np.abs(o1 - o2)) < 1e-13
        assert np.max(np.abs((l2 - l1) - shift)) < 1e-12


def test_rows_sample_matches_full():
    q, k, v, _ = _rand(1, 200, 2, 16, seed=10)
    out, lse = oracle.attention_fwd(q, k, v, causal=True)
    rows = [0, 1, 77, 199]
    ro, rl = oracle.attention_rows_fwd(q, k, v, 0, 1, rows, causal=True)
    assert np.max(np.abs(ro - out[0, rows, 1, :])) < 1e-14
    assert np.max(np.abs(rl - lse[0, 1, rows])) < 1e-14


def test_rows_dq_matches_full_backward():
    q, k, v, dout = _rand(1, 150, 2, 8, seed=14)
    for causal in (False, True):
        dq, _, _ = oracle.attention_bwd(q, k, v, dout, causal)
        rows = [0, 3, 149]
        got = oracle.attention_rows_dq(q, k, v, dout, 0, 1, rows, causal)
        assert np.max(np.abs(got - dq[0, rows, 1, :])) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_cols_dkdv_matches_full_backward(causal, monkeypatch):
    q, k, v, dout = _rand(1, 150, 2, 8, seed=15)
    _, dk, dv = oracle.attention_bwd(q, k, v, dout, causal)
    cols = [0, 7, 64, 148, 149]
    # several row blocks of a few rows each (the block size only bounds memory)
    for budget in (oatt._COL_BLOCK_VALUES, 6 * 150 + 5):
        monkeypatch.setattr(oatt, "_COL_BLOCK_VALUES", budget)
        gk, gv = oracle.attention_cols_dkdv(q, k, v, dout, 0, 1, cols, causal)
        assert np.max(np.abs(gk - dk[0, cols, 1, :])) < 1e-13
        assert np.max(np.abs(gv - dv[0, cols, 1, :])) < 1e-13


def test_cols_dkdv_matches_library_autograd():
    """The sampled key columns against torch's library attention and its autograd."""
    q, k, v, dout = _rand(1, 90, 2, 16, seed=16)
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).requires_grad_()
                  for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    o.backward(torch.from_numpy(np.ascontiguousarray(dout.transpose(0, 2, 1, 3))))
    cols = [3, 45, 80, 89]
    for h in range(2):
        gk, gv = oracle.attention_cols_dkdv(q, k, v, dout, 0, h, cols, causal=True)
        assert np.max(np.abs(gk - tk.grad.numpy()[0, h, cols, :])) < 1e-12
        assert np.max(np.abs(gv - tv.grad.numpy()[0, h, cols, :])) < 1e-12


def test_planted_unmasked_late_column_is_caught():
    """A column after a row's position must get nothing from that row: summing the
    unmasked terms instead fails the library pin."""
    q, k, v, dout = _rand(1, 40, 1, 8, seed=17)
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).requires_grad_()
                  for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    o.backward(torch.from_numpy(np.ascontiguousarray(dout.transpose(0, 2, 1, 3))))
    cols = [10, 30]
    right = oracle.attention_cols_dkdv(q, k, v, dout, 0, 0, cols, causal=True)
    # the non-causal column terms on causal probabilities would be the plausible slip
    wrong = oracle.attention_cols_dkdv(q, k, v, dout, 0, 0, cols, causal=False)
    want = tv.grad.numpy()[0, 0, cols, :]
    assert np.max(np.abs(right[1] - want)) < 1e-12
    assert np.max(np.abs(wrong[1] - want)) > 1e-3


def _loss(q, k, v, dout, causal):
    out, _ = oracle.attention_fwd(q, k, v, causal)
    return float(np.sum(out * dout))


def _fd_rel_errors(q, k, v, dout, causal, eps=1e-6):
    """Relative Frobenius error of the oracle's gradients against central differences
    of f = sum(dout * out)."""
    grads = oracle.attention_bwd(q, k, v, dout, causal)
    errs = {}
    for n, (name, x) in enumerate((("q", q), ("k", k), ("v", v))):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            a_p = dict(q=q, k=k, v=v); a_p[name] = xp
            a_m = dict(q=q, k=k, v=v); a_m[name] = xm
            num[idx] = (_loss(a_p["q"], a_p["k"], a_p["v"], dout, causal)
                        - _loss(a_m["q"], a_m["k"], a_m["v"], dout, causal)) / (2 * eps)
        errs[name] = np.linalg.norm(num - grads[n]) / np.linalg.norm(grads[n])
    return errs


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    q, k, v, dout = _rand(1, 12, 1, 4, seed=11)
    errs = _fd_rel_errors(q, k, v, dout, causal)
    assert max(errs.values()) < 1e-7, errs


@pytest.mark.parametrize("causal", [False, True])
def test_backward_closed_form_sums(causal):
    q, k, v, dout = _rand(2, 64, 2, 8, seed=12)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal)
    # every row of dS sums to 0 (rows of p sum to 1), so sum_c dK_c = 0
    assert np.max(np.abs(dk.sum(axis=1))) < 1e-12
    # sum_c p_rc = 1, so sum_c dV_c = sum_r dO_r
    assert np.max(np.abs(dv.sum(axis=1) - dout.sum(axis=1))) < 1e-12


def test_backward_matches_library_autograd():
    q, k, v, dout = _rand(1, 70, 2, 8, seed=13)
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).requires_grad_()
                  for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    o.backward(torch.from_numpy(np.ascontiguousarray(dout.transpose(0, 2, 1, 3))))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal=True)
    for g, t in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.max(np.abs(g - t.grad.numpy().transpose(0, 2, 1, 3))) < 1e-12


# ---- planted mistakes: each must be caught by one of the pins above -------------

def test_planted_mask_direction_is_caught(monkeypatch):
    good = oatt._scores

    def flipped(Qr, K, r0, causal, scale):
        s = scale * (Qr @ K.T)
        if causal:
            rows = np.arange(r0, r0 + Qr.shape[0])[:, None]
            cols = np.arange(K.shape[0])[None, :]
            s = np.where(cols < rows, -np.inf, s)     # wrong direction
        return s

    monkeypatch.setattr(oatt, "_scores", flipped)
    q, k, v, _ = _rand(1, 37, 2, 8, seed=1)
    out, _ = oracle.attention_fwd(q, k, v, True)
    assert not np.allclose(out, _sdpa(q, k, v, True), atol=1e-6)
    monkeypatch.setattr(oatt, "_scores", good)


def test_planted_missing_scale_is_caught():
    q, k, v, _ = _rand(1, 37, 2, 8, seed=1)
    out, _ = oracle.attention_fwd(q, k, v, False, scale=1.0)
    assert not np.allclose(out, _sdpa(q, k, v, False), atol=1e-6)


def test_planted_dropped_d_term_is_caught(monkeypatch):
    def no_d_term(p, Qr, K, V, dOr, scale):
        dS = p * (dOr @ V.T) * scale                  # forgets "- D"
        return dS @ K, dS.T @ Qr, p.T @ dOr

    monkeypatch.setattr(oatt, "_grad_rows", no_d_term)
    q, k, v, dout = _rand(1, 10, 1, 4, seed=11)
    errs = _fd_rel_errors(q, k, v, dout, causal=True)
    assert errs["q"] > 1e-2 and errs["k"] > 1e-2


def test_planted_transposed_p_is_caught(monkeypatch):
    def p_not_transposed(p, Qr, K, V, dOr, scale):
        O = p @ V
        Dr = np.sum(dOr * O, axis=1, keepdims=True)
        dS = p * (dOr @ V.T - Dr) * scale
        return dS @ K, dS.T @ Qr, p @ dOr             # p instead of p^T
    monkeypatch.setattr(oatt, "_grad_rows", p_not_transposed)
    q, k, v, dout = _rand(1, 10, 1, 4, seed=11)
    errs = _fd_rel_errors(q, k, v, dout, causal=False)
    assert errs["v"] > 1e-2
