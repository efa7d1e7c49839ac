"""Exact softmax attention in fp64, written from its definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition (labhub "Ring Attention 論文分析", section "標準 Self-Attention のメモリ
問題": the score matrix is Q K^T / sqrt(d_k), followed by a softmax over keys and a
product with V; the causal rule of section "Causal Masking の処理": a query never
attends to a later token).  For one (batch, head), in natural token order:

    s[r, c]  = scale * q_r . k_c                       (scale = 1/sqrt(D) by default)
    masked   : c > r when causal (strict upper triangle, excluded from the softmax)
    lse[r]   = ln sum_{c unmasked} exp(s[r, c])        (natural log)
    p[r, c]  = exp(s[r, c] - lse[r])                   (0 where masked)
    out[r]   = sum_c p[r, c] v_c

Backward (labhub, section "逆伝播での KV 再循環": D = rowsum(dO * O); dV = P^T dO;
dP = dO V^T; dS = P * (dP - D) * scale; dQ = dS K; dK = dS^T Q):

    D[r]     = dO_r . O_r
    dP[r, c] = dO_r . v_c
    dS[r, c] = p[r, c] * (dP[r, c] - D[r]) * scale
    dQ_r = sum_c dS[r, c] k_c ;  dK_c = sum_r dS[r, c] q_r ;  dV_c = sum_r p[r, c] dO_r

Implementation: query rows are processed in blocks against ALL keys with an exact
two-pass (max, then sum) softmax over the full row.  There is no online merge and no
ring here; those live in ``ring.py`` and in the CUDA path.  Keys after the last row of
a block are dropped before the product when causal: they are all masked for that
block, so this only skips exact zeros.

Tensors are float64 NumPy arrays laid out [B, L, H, D] (tokens in natural order);
lse is [B, H, L].
"""

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_ROW_BLOCK = 256
# attention_cols_dkdv: values in one block's score matrix (bounds its memory)
_COL_BLOCK_VALUES = 1 << 26


def default_scale(head_dim):
    """1/sqrt(d_k), the scale used on every page (e.g. labhub section "ブロック単位の
    分割戦略", and the ``scale`` argument of the ring forward)."""
    return 1.0 / math.sqrt(head_dim)


def _check(q, k, v):
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, L, H, D] shape")
    return q.shape


def _scores(Qr, K, r0, causal, scale):
    """Scaled scores of query rows r0..r0+R-1 against keys 0..C-1, masked."""
    R = Qr.shape[0]
    C = K.shape[0]
    s = scale * (Qr @ K.T)
    if causal:
        rows = np.arange(r0, r0 + R)[:, None]
        cols = np.arange(C)[None, :]
        s = np.where(cols > rows, -np.inf, s)
    return s


def _softmax_rows(s):
    """Exact two-pass softmax over full rows: returns (p, lse).

    A row with no visible key (every score -inf) gets p = 0 and lse = -inf.  Only that
    case is guarded: a NaN score (from a NaN input) makes its whole row's p and lse NaN,
    as the arithmetic gives."""
    m = np.max(s, axis=1, keepdims=True)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    with np.errstate(invalid="ignore"):
        e = np.exp(s - m_safe)
    tot = np.sum(e, axis=1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot == 0, -np.inf, m_safe + np.log(tot))
        p = np.where(tot == 0, 0.0, e / tot)
    return p, lse[:, 0]


def attention_fwd(q, k, v, causal, scale=None):
    """Forward pass. Returns (out [B,L,H,D], lse [B,H,L]) in float64."""
    B, L, H, D = _check(q, k, v)
    if scale is None:
        scale = default_scale(D)
    out = np.zeros((B, L, H, D))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            Q, K, V = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :]
            for r0 in range(0, L, _ROW_BLOCK):
                r1 = min(L, r0 + _ROW_BLOCK)
                C = r1 if causal else L
                s = _scores(Q[r0:r1], K[:C], r0, causal, scale)
                p, l_ = _softmax_rows(s)
                out[b, r0:r1, h, :] = p @ V[:C]
                lse[b, h, r0:r1] = l_
    return out, lse


def attention_rows_fwd(q, k, v, b, h, rows, causal, scale=None):
    """Forward for a few sampled query rows of one (batch, head).

    Used where the full problem is too large for the CPU: each row costs O(L*D).
    Returns (out [len(rows), D], lse [len(rows)]).
    """
    D = q.shape[3]
    if scale is None:
        scale = default_scale(D)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), D))
    lse = np.zeros(len(rows))
    for n, r in enumerate(rows):
        C = int(r) + 1 if causal else k.shape[1]
        K = np.asarray(k[b, :C, h, :], dtype=np.float64)
        V = np.asarray(v[b, :C, h, :], dtype=np.float64)
        s = _scores(np.asarray(q[b, r:r + 1, h, :], dtype=np.float64), K, int(r),
                    causal, scale)
        p, l_ = _softmax_rows(s)
        out[n] = (p @ V)[0]
        lse[n] = l_[0]
    return out, lse


def attention_rows_dq(q, k, v, dout, b, h, rows, causal, scale=None):
    """dQ for a few sampled query rows of one (batch, head), O(L*D) per row.

    Row r needs only its own softmax row: dQ_r = sum_c dS[r, c] k_c with
    dS[r, c] = p[r, c] (dO_r . v_c - dO_r . O_r) * scale.  Returns [len(rows), D].
    """
    D = q.shape[3]
    if scale is None:
        scale = default_scale(D)
    out = np.zeros((len(rows), D))
    for n, r in enumerate(np.asarray(rows, dtype=np.int64)):
        C = int(r) + 1 if causal else k.shape[1]
        K = np.asarray(k[b, :C, h, :], dtype=np.float64)
        V = np.asarray(v[b, :C, h, :], dtype=np.float64)
        Qr = np.asarray(q[b, r:r + 1, h, :], dtype=np.float64)
        dOr = np.asarray(dout[b, r:r + 1, h, :], dtype=np.float64)
        p, _ = _softmax_rows(_scores(Qr, K, int(r), causal, scale))
        gq, _, _ = _grad_rows(p, Qr, K, V, dOr, scale)
        out[n] = gq[0]
    return out


def attention_cols_dkdv(q, k, v, dout, b, h, cols, causal, scale=None, threads=None):
    """dK and dV for a few sampled key columns of one (batch, head).

    Used where the full backward is too large for the CPU.  By the formulas in the module
    docstring, key column c collects one term from every query row r that sees it (r >= c
    when causal, every row otherwise):
        dK_c = sum_r dS[r, c] q_r ,   dV_c = sum_r p[r, c] dO_r ,
    and each such row needs its own whole softmax row (p[r, c] = exp(s[r, c] - lse_r)) and
    its output O_r (for D_r = dO_r . O_r).  The cost is O(R * L * D) for the R rows that see
    the earliest sampled column, so the last columns of a long sequence are cheap.

    The rows are taken in independent blocks (each block's terms are computed on its own
    thread: NumPy releases the interpreter lock inside its array operations); the blocks'
    terms are then added in row order.  Returns (dk [len(cols), D], dv [len(cols), D]).
    """
    L, D = q.shape[1], q.shape[3]
    if scale is None:
        scale = default_scale(D)
    cols = np.asarray(cols, dtype=np.int64)
    K = np.asarray(k[b, :, h, :], dtype=np.float64)
    V = np.asarray(v[b, :, h, :], dtype=np.float64)
    Kc, Vc = K[cols], V[cols]
    r_first = int(cols.min()) if causal else 0
    step = max(1, _COL_BLOCK_VALUES // L)         # rows per block

    def block_terms(r0):
        r1 = min(L, r0 + step)
        C = r1 if causal else L
        Qr = np.asarray(q[b, r0:r1, h, :], dtype=np.float64)
        dOr = np.asarray(dout[b, r0:r1, h, :], dtype=np.float64)
        s = scale * (Qr @ K[:C].T)
        if causal:      # c > r happens only among the block's own keys [r0, r1)
            own = s[:, r0:C]
            own[np.triu_indices(r1 - r0, 1)] = -np.inf
        p, _ = _softmax_rows(s)
        Dr = np.sum(dOr * (p @ V[:C]), axis=1, keepdims=True)
        # p at the sampled columns; a column at or past C is masked for every row here
        pc = np.zeros((r1 - r0, len(cols)))
        seen = cols < C
        pc[:, seen] = p[:, cols[seen]]
        dSc = pc * (dOr @ Vc.T - Dr) * scale
        return dSc.T @ Qr, pc.T @ dOr

    starts = list(range(r_first, L, step))
    n_thr = threads or min(len(starts), len(os.sched_getaffinity(0)), 4)
    if n_thr > 1:
        with ThreadPoolExecutor(max_workers=n_thr) as ex:
            parts = list(ex.map(block_terms, starts))
    else:
        parts = [block_terms(r0) for r0 in starts]
    dk = np.zeros((len(cols), D))
    dv = np.zeros((len(cols), D))
    for gk, gv in parts:
        dk += gk
        dv += gv
    return dk, dv


def attention_bwd(q, k, v, dout, causal, scale=None):
    """Backward pass by the formulas in the module docstring.

    The softmax is recomputed from q, k (the pages' recompute strategy, labhub
    section "チェックポインティング戦略"), and O is the exact fp64 output.
    Returns (dq, dk, dv) in float64, [B, L, H, D].
    """
    B, L, H, D = _check(q, k, v)
    if scale is None:
        scale = default_scale(D)
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dv = np.zeros_like(v, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            Q, K, V = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :]
            dO = dout[b, :, h, :]
            for r0 in range(0, L, _ROW_BLOCK):
                r1 = min(L, r0 + _ROW_BLOCK)
                C = r1 if causal else L
                s = _scores(Q[r0:r1], K[:C], r0, causal, scale)
                p, _ = _softmax_rows(s)
                gq, gk, gv = _grad_rows(p, Q[r0:r1], K[:C], V[:C], dO[r0:r1], scale)
                dq[b, r0:r1, h, :] = gq
                dk[b, :C, h, :] += gk
                dv[b, :C, h, :] += gv
    return dq, dk, dv


def _grad_rows(p, Qr, K, V, dOr, scale):
    """Gradient contributions of one block of query rows (formulas above)."""
    O = p @ V
    Dr = np.sum(dOr * O, axis=1, keepdims=True)
    dP = dOr @ V.T
    dS = p * (dP - Dr) * scale
    return dS @ K, dS.T @ Qr, p.T @ dOr


def brute_force_fwd(q, k, v, causal, scale=None):
    """Pure-Python triple loop over (row, key, dim) for tiny inputs.

    Independent of NumPy's matrix products; used to pin ``attention_fwd``'s
    indexing (which axis is the token axis, the mask direction, the lse base).
    """
    B, L, H, D = _check(q, k, v)
    if scale is None:
        scale = default_scale(D)
    out = np.zeros((B, L, H, D))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            for r in range(L):
                keys = range(r + 1) if causal else range(L)
                sc = []
                for c in keys:
                    dot = 0.0
                    for d in range(D):
                        dot += float(q[b, r, h, d]) * float(k[b, c, h, d])
                    sc.append(scale * dot)
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = math.fsum(w)
                lse[b, h, r] = mx + math.log(tot)
                for d in range(D):
                    acc = 0.0
                    for wi, c in zip(w, keys):
                        acc += wi * float(v[b, c, h, d])
                    out[b, r, h, d] = acc / tot
    return out, lse
