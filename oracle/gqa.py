"""Grouped-query attention in fp64: fewer key/value heads than query heads.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: labhub "Ring Attention 論文分析", comparison section "比較分析: Ring Attention vs
Sequence Parallelism vs Tensor Parallelism" (table row "GQA/MQA 互換性" and the analysis
that follows it): ring attention works unchanged when several query heads share one
key/value head (GQA; MQA is the case of a single KV head), because the ring splits the
sequence, not the heads.  The page does not spell the grouping out; the reading taken here
is the usual one:

    H_q query heads, H_kv key/value heads, H_kv divides H_q, G = H_q / H_kv;
    query head h attends with key/value head h // G (G consecutive query heads share one).

Forward: out[:, :, h], lse[:, h] = attention(q[:, :, h], k[:, :, h // G], v[:, :, h // G]).
Backward: dq per query head as in plain attention; the gradient of a shared key/value
head is the sum over the G query heads that read it:
    dk[:, :, j] = sum_{h : h // G == j} dk_h ,   dv likewise.

Implementation: each KV head is repeated G times along the head axis (so that head h of the
expanded tensors is KV head h // G), the plain oracle runs on the expanded tensors, and the
per-query-head dK, dV are summed over each group.
"""

import numpy as np

from .attention import attention_bwd, attention_cols_dkdv, attention_fwd


def group_size(q_heads, kv_heads):
    if kv_heads < 1 or q_heads % kv_heads:
        raise ValueError("kv heads (%d) must divide query heads (%d)" % (kv_heads, q_heads))
    return q_heads // kv_heads


def _expand(x, G):
    return np.repeat(x, G, axis=2)      # head h of the result is head h // G of x


def gqa_fwd(q, k, v, causal, scale=None):
    """q [B, L, H_q, D]; k, v [B, L, H_kv, D].  Returns (out [B, L, H_q, D], lse [B, H_q, L])."""
    G = group_size(q.shape[2], k.shape[2])
    return attention_fwd(q, _expand(k, G), _expand(v, G), causal, scale)


def gqa_bwd(q, k, v, dout, causal, scale=None):
    """Returns (dq [B, L, H_q, D], dk [B, L, H_kv, D], dv [B, L, H_kv, D])."""
    G = group_size(q.shape[2], k.shape[2])
    dq, dk_e, dv_e = attention_bwd(q, _expand(k, G), _expand(v, G), dout, causal, scale)
    B, L, Hkv, D = k.shape
    return dq, dk_e.reshape(B, L, Hkv, G, D).sum(3), dv_e.reshape(B, L, Hkv, G, D).sum(3)


def gqa_cols_dkdv(q, k, v, dout, b, hk, cols, causal, scale=None):
    """dK and dV of key/value head hk at a few sampled key columns: the sum, over the G
    query heads h = hk * G + g that read that head, of each query head's column terms
    (``attention_cols_dkdv``).  Returns (dk [len(cols), D], dv [len(cols), D])."""
    G = group_size(q.shape[2], k.shape[2])
    dk = dv = 0.0
    for g in range(G):
        h = hk * G + g
        gk, gv = attention_cols_dkdv(q[:, :, h:h + 1], k[:, :, hk:hk + 1], v[:, :, hk:hk + 1],
                                     dout[:, :, h:h + 1], b, 0, cols, causal, scale)
        dk, dv = dk + gk, dv + gv
    return dk, dv
