"""GPU parity of the blockwise transformer layer (ra_linear, ra_layernorm, ra_bpt_fwd
through the C ABI) against the fp64 oracle on the same bf16 inputs and weights.

Tolerances (derived from the arithmetic): a Linear with fp32 accumulation agrees with fp64
to ~K * 2^-24 relative, so a bf16 output is bounded by its own rounding, 2^-8 relative
(+1e-3 absolute for values near zero), and an fp32 output by 1e-3 absolute.  The layer
rounds six intermediates to bf16 (Q, K, V, the attention output, LN1's output, the GELU
output), each a relative 2^-9; through the normalisations that is a relative error of
about sqrt(6) * 2^-9 = 5e-3 per element, so the test bounds the relative Frobenius error
by 1e-2 and the largest element error by 5e-2 (outputs are O(1), |y| < 6).
"""

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300.synthetic import make_bpt_weights, make_inputs

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("M,K,N", [(384, 192, 512), (256, 4096, 256), (128, 64, 768)])
@pytest.mark.parametrize("epi", ["bias", "bias_gelu", "bias_residual"])
def test_linear_parity(M, K, N, epi):
    g = torch.Generator().manual_seed(M + K + N)
    x = torch.randn((M, K), generator=g).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g) / K ** 0.5).to(torch.bfloat16)
    b = torch.randn(N, generator=g)
    res = torch.randn((M, N), generator=g).to(torch.bfloat16)
    ref = oracle.bpt.linear(_f64(x), _f64(w), _f64(b))
    if epi == "bias_gelu":
        ref = oracle.gelu(ref)
    if epi == "bias_residual":
        ref = ref + _f64(res)
    out = era.ra_linear(x.cuda(), w.cuda(), b.cuda(), epi,
                        residual=res.cuda() if epi == "bias_residual" else None)
    torch.cuda.synchronize()
    got = _f64(out)
    if epi == "bias_residual":
        assert out.dtype == torch.float32
        assert np.max(np.abs(got - ref)) <= 1e-3
    else:
        assert out.dtype == torch.bfloat16
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3)


@pytest.mark.parametrize("d", [512, 4096, 8192])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_layernorm_parity(d, out_dtype):
    g = torch.Generator().manual_seed(d)
    x = torch.randn((37, d), generator=g) * 3.0 + 1.5
    ga = 1.0 + 0.1 * torch.randn(d, generator=g)
    be = 0.1 * torch.randn(d, generator=g)
    ref = oracle.layer_norm(_f64(x), _f64(ga), _f64(be))
    got = _f64(era.ra_layernorm(x.cuda(), ga.cuda(), be.cuda(), 1e-5, out_dtype))
    if out_dtype == torch.float32:
        assert np.max(np.abs(got - ref)) <= 1e-4
    else:
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4)


def _layer_case(B, L, H, d_ff, seed):
    d = H * 128
    x = make_inputs(B, L, 1, d, seed, with_dout=False)[0].view(B, L, d)
    w = make_bpt_weights(d, d_ff, seed + 1)
    ref = oracle.bpt_layer_fwd(_f64(x), {k: _f64(v) for k, v in w.items()}, H, True)
    return x, w, ref


@pytest.mark.parametrize("layout", ["striped", "zigzag", "contiguous"])
def test_bpt_layer_parity(layout):
    B, L, H, d_ff, P = 1, 1024, 4, 1024, 4
    x, w, ref = _layer_case(B, L, H, d_ff, seed=50)
    wd = {k: v.cuda() for k, v in w.items()}
    out = era.ra_bpt_fwd(x.cuda(), wd, H, P, 128, layout, True, block_rows=256,
                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    got = _f64(out)
    err = got - ref
    assert np.linalg.norm(err) / np.linalg.norm(ref) <= 1e-2
    assert np.max(np.abs(err)) <= 5e-2


def test_bpt_layer_noncausal_contiguous():
    B, L, H, d_ff, P = 2, 512, 4, 512, 2
    d = H * 128
    x = make_inputs(B, L, 1, d, 70, with_dout=False)[0].view(B, L, d)
    w = make_bpt_weights(d, d_ff, 71)
    ref = oracle.bpt_layer_fwd(_f64(x), {k: _f64(v) for k, v in w.items()}, H, False)
    out = era.ra_bpt_fwd(x.cuda(), {k: v.cuda() for k, v in w.items()}, H, P, 128, "contiguous",
                         False, out_dtype=torch.float32)
    torch.cuda.synchronize()
    err = _f64(out) - ref
    assert np.linalg.norm(err) / np.linalg.norm(ref) <= 1e-2
    assert np.max(np.abs(err)) <= 5e-2


def test_bpt_blocking_does_not_change_the_result():
    B, L, H, d_ff, P = 2, 1024, 4, 512, 4
    x, w, ref = _layer_case(B, L, H, d_ff, seed=60)
    xd, wd = x.cuda(), {k: v.cuda() for k, v in w.items()}
    outs = [era.ra_bpt_fwd(xd, wd, H, P, 128, "zigzag", True, block_rows=br) for br in (0, 128, 640)]
    torch.cuda.synchronize()
    # every row's projections, normalisations and feed-forward are computed the same way
    # whatever block holds it: bit-identical
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    got = _f64(outs[0])
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-2


def test_bpt_fullsize_sampled_rows():
    """The 32k layer workload in the configuration bench.py times (zigzag, block_rows
    16384, bf16 output), checked on sampled rows: both ends, the block boundary, interior
    rows.  The oracle computes K and V of every row and the layer for the sampled rows."""
    from exact_blockwise_ring_gb300.synthetic import WORKLOADS, SEEDS
    wl = WORKLOADS["32k-bpt"]
    B, L, H, D, P, blk = (wl["batch"], wl["seq_len"], wl["heads"], wl["head_dim"], wl["P"],
                          wl["block"])
    d, d_ff, br = H * D, wl["d_ff"], wl["block_rows"]
    x = make_inputs(B, L, 1, d, SEEDS["32k-bpt"], with_dout=False)[0].view(B, L, d)
    w = make_bpt_weights(d, d_ff, SEEDS["32k-bpt"] + 1)
    out = era.ra_bpt_fwd(x.cuda(), {k: v.cuda() for k, v in w.items()}, H, P, blk, "zigzag",
                         True, block_rows=br)
    torch.cuda.synchronize()
    rows = [0, 1, br - 1, br, L // 3 + 7, L - 1]
    ref = oracle.bpt_layer_rows(_f64(x), {k: _f64(v) for k, v in w.items()}, H, True, 0, rows)
    got = _f64(out[0, rows])
    err = got - ref
    assert np.linalg.norm(err) / np.linalg.norm(ref) <= 1e-2
    assert np.all(np.abs(err) <= 5e-2 + 2.0 ** -8 * np.abs(ref))


def _layer_grads_case(B, L, H, d_ff, seed, Hkv=None, hd=128):
    d = H * hd
    x = make_inputs(B, L, 1, d, seed, with_dout=False)[0].view(B, L, d)
    dout = make_inputs(B, L, 1, d, seed + 1, with_dout=False)[0].view(B, L, d)
    w = make_bpt_weights(d, d_ff, seed + 2, d_kv=None if Hkv is None else Hkv * hd)
    ref = oracle.bpt_layer_bwd(_f64(x), {k: _f64(v) for k, v in w.items()}, H, True, _f64(dout))
    return x, dout, w, ref


@pytest.mark.parametrize("layout,B,block_rows", [("striped", 1, 256), ("zigzag", 2, 384),
                                                 ("contiguous", 1, 0)])
def test_bpt_backward_parity(layout, B, block_rows):
    """Every gradient within 2e-2 relative Frobenius error of the fp64 chain rule (as for the
    attention's gradients).  The K bias's gradient is exactly zero (adding a vector to every
    key shifts each query's scores by a constant), so it is checked as that identity."""
    H, d_ff, P, L = 4, 1024, 4, 1024
    x, dout, w, ref = _layer_grads_case(B, L, H, d_ff, seed=80)
    wd = {k: v.cuda() for k, v in w.items()}
    ws = era.Workspace("cuda")
    era.ra_bpt_fwd(x.cuda(), wd, H, P, 128, layout, True, block_rows=block_rows, workspace=ws,
                   train=True)
    g = era.ra_bpt_bwd(x.cuda(), wd, dout.cuda(), H, P, 128, layout, True, block_rows=block_rows,
                       workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    errs = {}
    for n in ["x"] + [n for n in era.BPT_WEIGHTS if n != "bk"]:
        errs[n] = float(np.linalg.norm(_f64(g[n]) - ref[n]) / np.linalg.norm(ref[n]))
    assert max(errs.values()) <= 2e-2, errs
    assert float(np.linalg.norm(_f64(g["bk"]))) <= 2e-2 * float(np.linalg.norm(ref["bv"]))


@pytest.mark.parametrize("layout,Hkv", [("striped", None), ("zigzag", 4)])
def test_bpt_backward_head_dim_64(layout, Hkv):
    """The layer at head_dim 64 (8 heads, d_model 512; grouped-query 8:4 in one case): every
    gradient within 2e-2 relative Frobenius error of the fp64 chain rule."""
    H, d_ff, P, L = 8, 1024, 4, 1024
    x, dout, w, ref = _layer_grads_case(1, L, H, d_ff, seed=64, Hkv=Hkv, hd=64)
    wd = {k: v.cuda() for k, v in w.items()}
    ws = era.Workspace("cuda")
    era.ra_bpt_fwd(x.cuda(), wd, H, P, 128, layout, True, block_rows=512, workspace=ws,
                   train=True)
    g = era.ra_bpt_bwd(x.cuda(), wd, dout.cuda(), H, P, 128, layout, True, block_rows=512,
                       workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    errs = {n: float(np.linalg.norm(_f64(g[n]) - ref[n]) / np.linalg.norm(ref[n]))
            for n in ["x"] + [n for n in era.BPT_WEIGHTS if n != "bk"]}
    assert max(errs.values()) <= 2e-2, errs
    assert float(np.linalg.norm(_f64(g["bk"]))) <= 2e-2 * float(np.linalg.norm(ref["bv"]))


def test_bpt_autograd_and_blocking():
    """BptLayer through torch autograd gives ra_bpt_bwd's gradients; a different block size
    changes only the fp32 summation order of the weight gradients."""
    H, d_ff, P, L = 4, 512, 4, 1024
    x, dout, w, _ = _layer_grads_case(1, L, H, d_ff, seed=90)
    xd = x.cuda().requires_grad_(True)
    params = [w[n].cuda().requires_grad_(True) for n in era.BPT_WEIGHTS]
    out = era.BptLayer.apply(xd, (H, P, 128, "zigzag", True, 256), *params)
    out.backward(dout.cuda())
    wd = {n: p.detach() for n, p in zip(era.BPT_WEIGHTS, params)}
    ws = era.Workspace("cuda")
    out2 = era.ra_bpt_fwd(x.cuda(), wd, H, P, 128, "zigzag", True, block_rows=512, workspace=ws,
                          train=True)
    g = era.ra_bpt_bwd(x.cuda(), wd, dout.cuda(), H, P, 128, "zigzag", True, block_rows=512,
                       workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), out2)
    assert float((xd.grad.float() - g["x"].float()).abs().max()) <= 1e-2
    for n, p in zip(era.BPT_WEIGHTS, params):
        if n == "bk":                       # exactly zero in exact arithmetic: noise only
            continue
        ref = g[n].to(p.dtype).float()
        den = float(ref.norm()) or 1.0
        assert float((p.grad.float() - ref).norm()) <= 1e-2 * den + 1e-6, n


def test_bpt_backward_fullsize_identities():
    """The 32k layer workload's forward + backward in the configuration bench.py times,
    checked through identities that hold at any size: d ln2_b = sum over rows of dout;
    d ln2_g = sum over rows of dout * (out - ln2_b) / ln2_g (the normalised value, read
    back from the fp32 forward output); the K bias's gradient vanishes."""
    from exact_blockwise_ring_gb300.synthetic import WORKLOADS, SEEDS
    wl = WORKLOADS["32k-bpt"]
    B, L, H, D, P, blk = (wl["batch"], wl["seq_len"], wl["heads"], wl["head_dim"], wl["P"],
                          wl["block"])
    d, d_ff, br = H * D, wl["d_ff"], wl["block_rows"]
    dev = torch.device("cuda:0")
    x = make_inputs(B, L, 1, d, SEEDS["32k-bpt"], device=dev, with_dout=False)[0].view(B, L, d)
    dout = make_inputs(B, L, 1, d, SEEDS["32k-bpt"] + 2, device=dev,
                       with_dout=False)[0].view(B, L, d)
    w = make_bpt_weights(d, d_ff, SEEDS["32k-bpt"] + 1, device=dev)
    ws = era.Workspace(dev)
    out = era.ra_bpt_fwd(x, w, H, P, blk, "zigzag", True, block_rows=br, workspace=ws,
                         out_dtype=torch.float32, train=True)
    g = era.ra_bpt_bwd(x, w, dout, H, P, blk, "zigzag", True, block_rows=br, workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    do64 = dout.double().view(-1, d)
    want_b = do64.sum(0)
    assert float((g["ln2_b"].double() - want_b).norm() / want_b.norm()) <= 1e-4
    yhat = (out.double().view(-1, d) - w["ln2_b"].double()) / w["ln2_g"].double()
    want_g = (do64 * yhat).sum(0)
    assert float((g["ln2_g"].double() - want_g).norm() / want_g.norm()) <= 1e-3
    assert float(g["bk"].norm()) <= 2e-2 * float(g["bv"].norm())
    for n, t in g.items():
        assert torch.isfinite(t).all(), n


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_bpt_grouped_query_layer(layout):
    """K and V projected to 2 heads for 4 query heads: forward and backward against the
    oracle's layer with grouped-query attention."""
    B, L, H, Hkv, d_ff, P = 1, 1024, 4, 2, 1024, 4
    x, dout, w, ref = _layer_grads_case(B, L, H, d_ff, seed=95, Hkv=Hkv)
    w64 = {k: _f64(v) for k, v in w.items()}
    out_ref = oracle.bpt_layer_fwd(_f64(x), w64, H, True)
    wd = {k: v.cuda() for k, v in w.items()}
    ws = era.Workspace("cuda")
    out = era.ra_bpt_fwd(x.cuda(), wd, H, P, 128, layout, True, block_rows=512, workspace=ws,
                         out_dtype=torch.float32, train=True)
    g = era.ra_bpt_bwd(x.cuda(), wd, dout.cuda(), H, P, 128, layout, True, block_rows=512,
                       workspace=ws)
    torch.cuda.synchronize()
    ws.check()
    eo = _f64(out) - out_ref
    assert np.linalg.norm(eo) / np.linalg.norm(out_ref) <= 1e-2 and np.max(np.abs(eo)) <= 5e-2
    assert g["wk"].shape == w["wk"].shape and g["bv"].shape == w["bv"].shape
    errs = {n: float(np.linalg.norm(_f64(g[n]) - ref[n]) / np.linalg.norm(ref[n]))
            for n in ["x"] + [n for n in era.BPT_WEIGHTS if n != "bk"]}
    assert max(errs.values()) <= 2e-2, errs
    assert float(np.linalg.norm(_f64(g["bk"]))) <= 2e-2 * float(np.linalg.norm(ref["bv"]))
