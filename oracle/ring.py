"""fp64 emulator of the ring schedule with blockwise online softmax.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Used only to test invariants of the method (the ring result equals full attention,
striped permutation then unpermutation changes nothing, merged per-step partials equal
the fused result).  It follows the pages' steps in their order:

* For every shard i and ring step k = 0..P-1 the KV shard is j = (i - k) mod P
  (labhub, section "リングトポロジーと KV の循環"; vanos001 ring diagram).
* Inside a step, KV blocks of `block` keys are taken one by one (labhub, section
  "ブロック単位の分割戦略"): new_max = max(max, blockmax); correction =
  exp(max - new_max); sum = sum*correction + rowsum(exp(s - new_max));
  acc = acc*correction + exp(s - new_max) V.
* Causal mask by ORIGINAL token positions: key token c is visible to query token r iff
  c <= r.  For contiguous shards this is the pages' block rule (skip later blocks,
  triangular mask on the same block, no mask on earlier ones, labhub section
  "Causal Masking の処理"); for striped shards the pages give no mask, and the reading
  taken is the same position rule, which is what permutation equivariance (aibr.jp,
  section 3) requires.
* Guard: while a row has seen no visible key its max is -inf; then the correction is
  taken as 1 and the block's exponentials as 0 (the pages' code would form
  exp(-inf - (-inf)) = NaN there; labhub "限界" notes NaN/Inf from the online softmax).
* After the last step: out = acc / sum, lse = max + ln(sum).

``ring_partials`` returns one normalised partial (O_k, lse_k) per ring step, and
``merge_partials`` combines them: lse = ln sum_k exp(lse_k), O = sum_k exp(lse_k - lse)
O_k, skipping steps with lse_k = -inf.  The pages merge only as a running update
(the correction step above); this is the same update written for whole partials.
"""

import numpy as np

from .attention import default_scale
from .work import shard_tokens


def _online_block(state, s, Vb):
    m, l_, acc = state
    bmax = np.max(s, axis=1)
    m_new = np.maximum(m, bmax)
    seen = np.isfinite(m_new)
    m_ref = np.where(seen, m_new, 0.0)
    corr = np.where(np.isfinite(m), np.exp(m - m_ref), 1.0)
    e = np.where(seen[:, None], np.exp(s - m_ref[:, None]), 0.0)
    l_ = l_ * corr + e.sum(axis=1)
    acc = acc * corr[:, None] + e @ Vb
    return m_new, l_, acc


def _finish(state):
    m, l_, acc = state
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(l_[:, None] > 0, acc / l_[:, None], 0.0)
        lse = np.where(l_ > 0, m + np.log(l_), -np.inf)
    return out, lse


def _shard_steps(q, k, v, b, h, i, P, layout, causal, scale, block):
    """Yield (k, step_state) after each ring step for the queries of shard i."""
    L = q.shape[1]
    D = q.shape[3]
    q_tok = np.array(shard_tokens(i, L, P, layout))
    Q = q[b, q_tok, h, :]
    n = len(q_tok)
    for kk in range(P):
        j = (i - kk) % P
        k_tok = np.array(shard_tokens(j, L, P, layout))
        state = (np.full(n, -np.inf), np.zeros(n), np.zeros((n, D)))
        yield kk, j, q_tok, Q, k_tok, state


def ring_partials(q, k, v, P, layout, causal, block, scale=None):
    """Per-step partials. Returns (o_parts [P,B,L,H,D], lse_parts [P,B,H,L]).

    Partial k of a query row is attention restricted to the KV shard visited at ring
    step k by that row's shard; rows with no visible key there get lse = -inf, O = 0.
    """
    B, L, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    o_parts = np.zeros((P, B, L, H, D))
    lse_parts = np.full((P, B, H, L), -np.inf)
    for b in range(B):
        for h in range(H):
            for i in range(P):
                for kk, j, q_tok, Q, k_tok, state in _shard_steps(
                        q, k, v, b, h, i, P, layout, causal, scale, block):
                    K = k[b, k_tok, h, :]
                    V = v[b, k_tok, h, :]
                    for u0 in range(0, len(k_tok), block):
                        kt = k_tok[u0:u0 + block]
                        s = scale * (Q @ K[u0:u0 + block].T)
                        if causal:
                            s = np.where(kt[None, :] > q_tok[:, None], -np.inf, s)
                        state = _online_block(state, s, V[u0:u0 + block])
                    o, l_ = _finish(state)
                    o_parts[kk, b, q_tok, h, :] = o
                    lse_parts[kk, b, h, q_tok] = l_
    return o_parts, lse_parts


def merge_partials(o_parts, lse_parts):
    """Merge normalised partials: o_parts [n, ..., rows, D], lse_parts [n, ..., rows]
    with matching leading shapes in the layouts used above ([n,B,L,H,D], [n,B,H,L]).
    Returns (out [B,L,H,D], lse [B,H,L])."""
    lse_t = np.transpose(lse_parts, (0, 1, 3, 2))          # [n, B, L, H]
    mx = np.max(lse_t, axis=0)
    mx_safe = np.where(np.isfinite(mx), mx, 0.0)
    w = np.where(np.isfinite(lse_t), np.exp(lse_t - mx_safe), 0.0)
    tot = np.sum(w, axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, mx_safe + np.log(tot), -np.inf)
        wn = np.where(tot > 0, w / tot, 0.0)
    out = np.sum(wn[..., None] * o_parts, axis=0)
    return out, np.transpose(lse, (0, 2, 1))


def ring_fwd(q, k, v, P, layout, causal, block, scale=None):
    """Fused ring forward: one online-softmax state per shard carried over all P steps.
    Returns (out [B,L,H,D], lse [B,H,L])."""
    B, L, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    out = np.zeros((B, L, H, D))
    lse = np.full((B, H, L), -np.inf)
    for b in range(B):
        for h in range(H):
            for i in range(P):
                q_tok = np.array(shard_tokens(i, L, P, layout))
                Q = q[b, q_tok, h, :]
                n = len(q_tok)
                state = (np.full(n, -np.inf), np.zeros(n), np.zeros((n, D)))
                for kk in range(P):
                    j = (i - kk) % P
                    k_tok = np.array(shard_tokens(j, L, P, layout))
                    K = k[b, k_tok, h, :]
                    V = v[b, k_tok, h, :]
                    for u0 in range(0, n, block):
                        kt = k_tok[u0:u0 + block]
                        if causal and kt.min() > q_tok.max():
                            continue          # whole block after every query: skip
                        s = scale * (Q @ K[u0:u0 + block].T)
                        if causal:
                            s = np.where(kt[None, :] > q_tok[:, None], -np.inf, s)
                        state = _online_block(state, s, V[u0:u0 + block])
                o, l_ = _finish(state)
                out[b, q_tok, h, :] = o
                lse[b, h, q_tok] = l_
    return out, lse
