"""Pins for the oracle's Blockwise Parallel Transformer layer (CPU only).

References: torch's library modules in float64 (nn.Linear, nn.LayerNorm, nn.GELU with
its exact erf form, scaled_dot_product_attention), the page's own per-block loop (the
fusion must not change the result), the normal CDF for GELU, and the moments of a
LayerNorm output.  Planted mistakes (tanh GELU, unbiased variance, no first residual)
are shown to fail the library pin.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import bpt as obpt


def _weights(d, d_ff, seed, d_kv=None):
    rng = np.random.default_rng(seed)
    w = {}
    d_kv = d if d_kv is None else d_kv
    for name, (o, i) in (("wq", (d, d)), ("wk", (d_kv, d)), ("wv", (d_kv, d)), ("wo", (d, d)),
                         ("w1", (d_ff, d)), ("w2", (d, d_ff))):
        w[name] = rng.standard_normal((o, i)) / math.sqrt(i)
        w["b" + name[1:]] = 0.1 * rng.standard_normal(o)
    for ln in ("ln1", "ln2"):
        w[ln + "_g"] = 1.0 + 0.1 * rng.standard_normal(d)
        w[ln + "_b"] = 0.1 * rng.standard_normal(d)
    return w


def _torch_layer(x, w, n_heads, causal):
    """The same layer from torch's library modules, float64."""
    d = x.shape[-1]
    d_ff = w["w1"].shape[0]
    d_kv = w["wk"].shape[0]
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))   # noqa: E731
    lin = {}
    for name, (o, i) in (("q", (d, d)), ("k", (d_kv, d)), ("v", (d_kv, d)), ("o", (d, d)),
                         ("1", (d_ff, d)), ("2", (d, d_ff))):
        m = torch.nn.Linear(i, o, dtype=torch.float64)
        with torch.no_grad():
            m.weight.copy_(T(w["w" + name]))
            m.bias.copy_(T(w["b" + name]))
        lin[name] = m
    lns = []
    for ln in ("ln1", "ln2"):
        m = torch.nn.LayerNorm(d, eps=1e-5, dtype=torch.float64)
        with torch.no_grad():
            m.weight.copy_(T(w[ln + "_g"]))
            m.bias.copy_(T(w[ln + "_b"]))
        lns.append(m)
    xt = T(x)
    B, L, _ = x.shape
    dk = d // n_heads
    split = lambda t: t.view(B, L, t.shape[-1] // dk, dk).transpose(1, 2)   # noqa: E731
    with torch.no_grad():
        a = F.scaled_dot_product_attention(split(lin["q"](xt)), split(lin["k"](xt)),
                                           split(lin["v"](xt)), is_causal=causal,
                                           enable_gqa=d_kv != d)
        a = a.transpose(1, 2).reshape(B, L, d)
        h1 = lns[0](xt + lin["o"](a))
        f = lin["2"](torch.nn.GELU()(lin["1"](h1)))
        return lns[1](h1 + f).numpy()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,L,d,H,d_ff,Hkv", [(1, 64, 32, 2, 64, 2), (2, 96, 48, 3, 96, 3),
                                              (1, 128, 64, 1, 256, 1), (1, 64, 64, 4, 128, 2),
                                              (2, 48, 32, 4, 64, 1)])
def test_layer_matches_library_modules(causal, B, L, d, H, d_ff, Hkv):
    w = _weights(d, d_ff, seed=L + d, d_kv=Hkv * (d // H))
    x = np.random.default_rng(L).standard_normal((B, L, d))
    got = oracle.bpt_layer_fwd(x, w, H, causal)
    want = _torch_layer(x, w, H, causal)
    assert np.max(np.abs(got - want)) < 1e-10


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("block", [16, 32, 128])
@pytest.mark.parametrize("d_kv", [32, 16])
def test_blockwise_loop_equals_whole_sequence(causal, block, d_kv):
    w = _weights(32, 64, seed=3, d_kv=d_kv)
    x = np.random.default_rng(4).standard_normal((2, 128, 32))
    a = oracle.bpt_layer_fwd(x, w, 2, causal)
    b = oracle.bpt_layer_fwd_blocked(x, w, 2, causal, block)
    assert np.max(np.abs(a - b)) < 1e-11


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d_kv", [64, 32])
def test_sampled_rows_equal_the_whole_layer(causal, d_kv):
    w = _weights(64, 128, seed=8, d_kv=d_kv)
    x = np.random.default_rng(9).standard_normal((2, 96, 64))
    full = oracle.bpt_layer_fwd(x, w, 2, causal)
    rows = [0, 1, 37, 95]
    for b in range(2):
        got = oracle.bpt_layer_rows(x, w, 2, causal, b, rows)
        assert np.max(np.abs(got - full[b, rows])) < 1e-11


def test_gelu_is_z_times_normal_cdf():
    z = np.array([-3.0, -1.0, 0.0, 0.5, 1.0, 2.0, 6.0])
    # Phi(1) and Phi(-1) to 16 digits, Phi(0) = 1/2
    assert abs(oracle.gelu(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    assert abs(oracle.gelu(np.array([-1.0]))[0] + 0.15865525393145707) < 1e-15
    assert oracle.gelu(np.array([0.0]))[0] == 0.0
    from scipy.stats import norm
    assert np.max(np.abs(oracle.gelu(z) - z * norm.cdf(z))) < 1e-15


def test_layer_norm_moments():
    y = np.random.default_rng(5).standard_normal((7, 64)) * 3.0 + 2.0
    out = oracle.layer_norm(y, np.ones(64), np.zeros(64))
    var = y.var(axis=-1)
    assert np.max(np.abs(out.mean(axis=-1))) < 1e-14
    assert np.max(np.abs(out.var(axis=-1) - var / (var + 1e-5))) < 1e-12


def test_planted_mistakes_fail_the_library_pin(monkeypatch):
    w = _weights(32, 64, seed=6)
    x = np.random.default_rng(7).standard_normal((1, 64, 32))
    want = _torch_layer(x, w, 2, True)

    def tanh_gelu(z):
        return 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))

    def unbiased_ln(y, g, b, eps=1e-5):
        return (y - y.mean(-1, keepdims=True)) / np.sqrt(y.var(-1, ddof=1, keepdims=True) + eps) * g + b

    def no_residual(xb, ab, ww):
        h1 = obpt.layer_norm(obpt.linear(ab, ww["wo"], ww["bo"]), ww["ln1_g"], ww["ln1_b"])
        f = obpt.linear(obpt.gelu(obpt.linear(h1, ww["w1"], ww["b1"])), ww["w2"], ww["b2"])
        return obpt.layer_norm(h1 + f, ww["ln2_g"], ww["ln2_b"])

    for attr, fake in (("gelu", tanh_gelu), ("layer_norm", unbiased_ln),
                       ("_post_attention", no_residual)):
        with monkeypatch.context() as mp:
            mp.setattr(obpt, attr, fake)
            got = obpt.bpt_layer_fwd(x, w, 2, True)
        assert np.max(np.abs(got - want)) > 1e-6, attr


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hkv", [4, 2, 1])
def test_layer_backward_matches_torch_autograd(causal, Hkv):
    B, L, d, H, d_ff = 2, 48, 32, 4, 64
    w = _weights(d, d_ff, seed=11, d_kv=Hkv * (d // H))
    x = np.random.default_rng(12).standard_normal((B, L, d))
    dout = np.random.default_rng(13).standard_normal((B, L, d))
    got = oracle.bpt_layer_bwd(x, w, H, causal, dout)
    # the same layer from torch's library modules, gradients by autograd
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).requires_grad_(True)   # noqa: E731
    wt = {k: T(v) for k, v in w.items()}
    xt = T(x)
    split = lambda t: t.view(B, L, t.shape[-1] // (d // H), d // H).transpose(1, 2)   # noqa: E731
    lin = lambda t, n: F.linear(t, wt["w" + n], wt["b" + n])     # noqa: E731
    a = F.scaled_dot_product_attention(split(lin(xt, "q")), split(lin(xt, "k")),
                                       split(lin(xt, "v")), is_causal=causal, enable_gqa=Hkv != H)
    a = a.transpose(1, 2).reshape(B, L, d)
    h1 = F.layer_norm(xt + lin(a, "o"), (d,), wt["ln1_g"], wt["ln1_b"], 1e-5)
    y = F.layer_norm(h1 + lin(F.gelu(lin(h1, "1")), "2"), (d,), wt["ln2_g"], wt["ln2_b"], 1e-5)
    (y * torch.from_numpy(dout)).sum().backward()
    assert np.max(np.abs(got["x"] - xt.grad.numpy())) < 1e-10
    for name in obpt.WEIGHT_NAMES:
        ref = wt[name].grad.numpy()
        assert np.max(np.abs(got[name] - ref)) < 1e-10 * max(1.0, np.max(np.abs(ref))), name


def test_gelu_and_layer_norm_grads_by_finite_differences():
    rng = np.random.default_rng(14)
    z = rng.standard_normal(9) * 2
    h = 1e-6
    fd = (oracle.gelu(z + h) - oracle.gelu(z - h)) / (2 * h)
    assert np.max(np.abs(fd - oracle.gelu_grad(z))) < 1e-8
    y = rng.standard_normal((3, 16))
    g, b = 1 + 0.1 * rng.standard_normal(16), rng.standard_normal(16)
    dout = rng.standard_normal((3, 16))
    dy, dg, db = oracle.layer_norm_bwd(y, g, dout)
    f = lambda yy: float(np.sum(oracle.layer_norm(yy, g, b) * dout))   # noqa: E731
    for (r, c) in [(0, 0), (1, 7), (2, 15)]:
        yp, ym = y.copy(), y.copy()
        yp[r, c] += h
        ym[r, c] -= h
        assert abs((f(yp) - f(ym)) / (2 * h) - dy[r, c]) < 1e-7
