"""One Blockwise Parallel Transformer layer, forward and backward, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: labhub "Ring Attention 論文分析", section "BPT の Feedforward 融合": the layer
projects the input to Q, K, V, and then, one query block at a time, takes that block's
attention over all keys, applies the output projection, adds the block's input and
normalises, applies the feed-forward network (Linear, GELU, Linear), adds the normalised
value and normalises again, and writes the block's output.  Only the current block's
intermediates are ever held, which is the point of the fusion; the result is the plain
post-norm transformer layer.  Written out, for x [B, L, d]:

    Q = x Wq^T + bq,  K = x Wk^T + bk,  V = x Wv^T + bv          (Linear: y = x W^T + b)
    A = attention(Q, K, V) over n_heads heads of d_k = d / n_heads (head h = features
        [h d_k, (h+1) d_k)), causal or not, scale 1 / sqrt(d_k)
    h1 = LN1(x + A Wo^T + bo)
    out = LN2(h1 + (GELU(h1 W1^T + b1)) W2^T + b2)

    LN(y) = (y - mean(y)) / sqrt(var(y) + eps) * gamma + beta over the d features of a row,
            var the biased (population) variance, eps = 1e-5;
    GELU(z) = z * Phi(z) = z / 2 * (1 + erf(z / sqrt(2)))   (the exact form).

The page's layer shows no mask; the attention here takes the same `causal` switch as the
rest of this package.  With Wk, Wv of H_kv * d_k rows (H_kv dividing n_heads) the
attention is grouped-query (``gqa.py``); H_kv = n_heads is the plain layer.  Weights follow torch.nn.Linear's layout: W [out_features,
in_features].  ``bpt_layer_fwd`` computes the whole sequence at once;
``bpt_layer_fwd_blocked`` follows the page's loop over query blocks and is used by the
tests to show that the two agree (the fusion changes memory, not the result).
``bpt_layer_rows`` evaluates the same definition for a few output rows of a long sequence
(the keys and values of every earlier row, then the sampled rows only), for checks at
sizes where the whole layer is out of reach in fp64.  ``bpt_layer_bwd`` gives the gradients
of sum(out * dout) with respect to x and every parameter by the chain rule through the
steps above (the attention's own backward is ``attention_bwd``):
    LN backward: dy = rstd (dyh - mean(dyh) - yh mean(dyh yh)), dyh = dout g,
                 dg = sum dout yh, db = sum dout;
    Linear backward: dx = dy W, dW = dy^T x, db = sum dy;
    GELU backward: dz = df (Phi(z) + z phi(z)).
"""

import math

import numpy as np

from .attention import attention_fwd
from .gqa import gqa_bwd, gqa_fwd

LN_EPS = 1e-5

WEIGHT_NAMES = ("wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo", "w1", "b1", "w2", "b2",
                "ln1_g", "ln1_b", "ln2_g", "ln2_b")


def _erf(z):
    return np.vectorize(math.erf, otypes=[np.float64])(z)


def gelu(z):
    """Exact GELU, z * Phi(z)."""
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def layer_norm(y, g, b, eps=LN_EPS):
    mu = y.mean(axis=-1, keepdims=True)
    var = ((y - mu) ** 2).mean(axis=-1, keepdims=True)
    return (y - mu) / np.sqrt(var + eps) * g + b


def linear(x, w, b):
    return x @ w.T + b


def _heads(t, n_heads):
    B, L, d = t.shape
    return t.reshape(B, L, n_heads, d // n_heads)


def _kv_heads(w, d, n_heads):
    """Key/value heads: Wk is [H_kv * d_k, d] (grouped-query attention when H_kv < H)."""
    return w["wk"].shape[0] // (d // n_heads)


def _post_attention(xb, ab, w):
    """Output projection, residual, LN1, FFN, residual, LN2 for rows xb with attention ab."""
    h1 = layer_norm(xb + linear(ab, w["wo"], w["bo"]), w["ln1_g"], w["ln1_b"])
    f = linear(gelu(linear(h1, w["w1"], w["b1"])), w["w2"], w["b2"])
    return layer_norm(h1 + f, w["ln2_g"], w["ln2_b"])


def bpt_layer_fwd(x, w, n_heads, causal):
    """x [B, L, d] float64, w dict of float64 arrays (WEIGHT_NAMES).  Returns [B, L, d]."""
    B, L, d = x.shape
    hkv = _kv_heads(w, d, n_heads)
    q = _heads(linear(x, w["wq"], w["bq"]), n_heads)
    k = _heads(linear(x, w["wk"], w["bk"]), hkv)
    v = _heads(linear(x, w["wv"], w["bv"]), hkv)
    a, _ = gqa_fwd(q, k, v, causal)
    return _post_attention(x, a.reshape(B, L, d), w)


def bpt_layer_fwd_blocked(x, w, n_heads, causal, block_size):
    """The page's loop: per query block, attention over all keys, then the rest."""
    B, L, d = x.shape
    if L % block_size:
        raise ValueError("seq_len must be a multiple of block_size")
    q = linear(x, w["wq"], w["bq"])
    hkv = _kv_heads(w, d, n_heads)
    k = np.repeat(_heads(linear(x, w["wk"], w["bk"]), hkv), n_heads // hkv, axis=2)
    v = np.repeat(_heads(linear(x, w["wv"], w["bv"]), hkv), n_heads // hkv, axis=2)
    out = np.zeros_like(x)
    dk = d // n_heads
    for s in range(0, L, block_size):
        qb = _heads(q[:, s:s + block_size], n_heads)
        # attention of this block's queries over all keys: masked by original positions
        # (query s + r sees keys <= s + r when causal)
        sc = np.einsum("brhd,bchd->bhrc", qb, k) / math.sqrt(dk)
        if causal:
            r = np.arange(block_size)[:, None] + s
            c = np.arange(L)[None, :]
            sc = np.where(c <= r, sc, -np.inf)
        sc = sc - sc.max(axis=-1, keepdims=True)
        p = np.exp(sc)
        p /= p.sum(axis=-1, keepdims=True)
        ab = np.einsum("bhrc,bchd->brhd", p, v).reshape(B, block_size, d)
        out[:, s:s + block_size] = _post_attention(x[:, s:s + block_size], ab, w)
    return out


def bpt_layer_rows(x, w, n_heads, causal, b, rows):
    """Output rows `rows` of batch entry b of the layer, [len(rows), d]."""
    B, L, d = x.shape
    dk = d // n_heads
    rows = np.asarray(rows)
    last = int(rows.max()) + 1 if causal else L
    xb = x[b]
    hkv = _kv_heads(w, d, n_heads)
    kk = np.repeat(linear(xb[:last], w["wk"], w["bk"]).reshape(last, hkv, dk), n_heads // hkv, 1)
    vv = np.repeat(linear(xb[:last], w["wv"], w["bv"]).reshape(last, hkv, dk), n_heads // hkv, 1)
    qq = linear(xb[rows], w["wq"], w["bq"]).reshape(len(rows), n_heads, dk)
    a = np.zeros((len(rows), n_heads, dk))
    for n, r in enumerate(rows):
        c = int(r) + 1 if causal else L
        s = np.einsum("hd,chd->hc", qq[n], kk[:c]) / math.sqrt(dk)
        s -= s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=-1, keepdims=True)
        a[n] = np.einsum("hc,chd->hd", p, vv[:c])
    return _post_attention(xb[rows], a.reshape(len(rows), d), w)


def gelu_grad(z):
    """d GELU / dz = Phi(z) + z phi(z)."""
    return 0.5 * (1.0 + _erf(z / math.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / math.sqrt(2 * math.pi)


def layer_norm_bwd(y, g, dout, eps=LN_EPS):
    """Gradients of LN(y) = (y - mean) / sqrt(var + eps) * g + b over the last axis:
    returns (dy, dg, db) with dg, db summed over every leading axis."""
    mu = y.mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(((y - mu) ** 2).mean(axis=-1, keepdims=True) + eps)
    yh = (y - mu) * rstd
    dyh = dout * g
    dy = rstd * (dyh - dyh.mean(axis=-1, keepdims=True) - yh * (dyh * yh).mean(axis=-1, keepdims=True))
    lead = tuple(range(y.ndim - 1))
    return dy, (dout * yh).sum(axis=lead), dout.sum(axis=lead)


def _linear_bwd(xin, w, dy):
    """y = xin w^T + b: returns (dxin, dw, db) with the rows of every leading axis summed."""
    d2 = dy.reshape(-1, dy.shape[-1])
    x2 = xin.reshape(-1, xin.shape[-1])
    return dy @ w, d2.T @ x2, d2.sum(axis=0)


def bpt_layer_bwd(x, w, n_heads, causal, dout):
    """Gradients of sum(out * dout) for the layer of bpt_layer_fwd, by the chain rule:
    returns a dict with "x" and every name of WEIGHT_NAMES."""
    B, L, d = x.shape
    hkv = _kv_heads(w, d, n_heads)
    q = _heads(linear(x, w["wq"], w["bq"]), n_heads)
    k = _heads(linear(x, w["wk"], w["bk"]), hkv)
    v = _heads(linear(x, w["wv"], w["bv"]), hkv)
    a4, _ = gqa_fwd(q, k, v, causal)
    a = a4.reshape(B, L, d)
    y1 = x + linear(a, w["wo"], w["bo"])
    h1 = layer_norm(y1, w["ln1_g"], w["ln1_b"])
    z = linear(h1, w["w1"], w["b1"])
    f = gelu(z)
    y2 = h1 + linear(f, w["w2"], w["b2"])
    g = {}
    dy2, g["ln2_g"], g["ln2_b"] = layer_norm_bwd(y2, w["ln2_g"], dout)
    df, g["w2"], g["b2"] = _linear_bwd(f, w["w2"], dy2)
    dz = df * gelu_grad(z)
    dh1_f, g["w1"], g["b1"] = _linear_bwd(h1, w["w1"], dz)
    dh1 = dy2 + dh1_f
    dy1, g["ln1_g"], g["ln1_b"] = layer_norm_bwd(y1, w["ln1_g"], dh1)
    da, g["wo"], g["bo"] = _linear_bwd(a, w["wo"], dy1)
    dq, dk, dv = gqa_bwd(q, k, v, da.reshape(B, L, n_heads, d // n_heads), causal)
    dx = dy1.copy()
    for t, wn, bn in ((dq, "wq", "bq"), (dk, "wk", "bk"), (dv, "wv", "bv")):
        dxi, g[wn], g[bn] = _linear_bwd(x, w[wn], t.reshape(B, L, -1))
        dx += dxi
    g["x"] = dx
    return g
