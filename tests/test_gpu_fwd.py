"""GPU parity of the forward path (ra_fwd through the C ABI) against the fp64 oracle.

Tolerances: output max-abs 1e-2 with fp32 output, lse max-abs 1e-3.  With bf16 output
the bound adds bf16's own rounding of the exact value (2^-8 relative).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300.synthetic import WORKLOADS, SEEDS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3


def _case(B, L, H, D, seed):
    q, k, v = make_inputs(B, L, H, D, seed, device="cpu", with_dout=False)
    return (q, k, v), to_f64(q, k, v)


def _gpu_fwd(qkv, P, block, layout, causal, out_dtype=torch.float32, n_split=0,
             shard_work=False):
    q, k, v = (t.cuda() for t in qkv)
    res = era.ra_fwd(q, k, v, P, block, layout, causal, out_dtype=out_dtype, n_split=n_split,
                     shard_work=shard_work)
    torch.cuda.synchronize()
    return res


def _errs(out, lse, o_ref, l_ref):
    o = out.float().cpu().numpy()
    l_ = lse.cpu().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(l_), fin)
    return float(np.max(np.abs(o - o_ref))), float(np.max(np.abs(l_[fin] - l_ref[fin])))


SWEEP = [
    # B, L, H, D, P, block, layout, causal, n_split
    (2, 1024, 3, 128, 2, 128, "contiguous", True, 1),
    (2, 1024, 3, 128, 2, 128, "striped", True, 1),
    (1, 1024, 2, 128, 8, 128, "striped", True, 1),      # one 128-row tile per shard
    (1, 1024, 2, 128, 8, 128, "contiguous", True, 1),
    (1, 1536, 2, 128, 4, 128, "contiguous", True, 1),   # 3 tiles per shard: ragged pair
    (1, 1536, 2, 128, 4, 128, "striped", True, 1),
    (1, 2048, 2, 128, 4, 256, "striped", True, 1),
    (1, 2048, 2, 64, 4, 256, "contiguous", True, 1),
    (1, 2048, 2, 64, 4, 128, "striped", True, 1),
    (1, 1024, 1, 128, 1, 128, "contiguous", True, 1),   # P = 1: plain blockwise attention
    (1, 1024, 2, 128, 4, 128, "contiguous", False, 1),
    (1, 1024, 2, 128, 4, 128, "striped", False, 1),
    (1, 2048, 2, 128, 4, 128, "striped", True, 2),      # split into partials + merge
    (1, 2048, 2, 128, 4, 128, "contiguous", True, 4),
    (1, 2048, 2, 64, 4, 128, "striped", True, 4),
    (1, 1024, 2, 128, 2, 128, "zigzag", True, 1),       # 2 tiles per chunk
    (2, 2048, 3, 128, 4, 128, "zigzag", True, 1),
    (1, 1536, 2, 128, 2, 128, "zigzag", True, 1),       # 3 tiles per chunk: a pair straddles
    (1, 2048, 2, 64, 4, 256, "zigzag", True, 1),
    (1, 2048, 2, 128, 4, 128, "zigzag", True, 2),
    (1, 1024, 2, 128, 4, 128, "zigzag", False, 1),
]


@pytest.mark.parametrize("B,L,H,D,P,block,layout,causal,n_split", SWEEP)
def test_fwd_parity_sweep(B, L, H, D, P, block, layout, causal, n_split):
    qkv, (q64, k64, v64) = _case(B, L, H, D, seed=L + 7 * H + D + P)
    o_ref, l_ref = oracle.attention_fwd(q64, k64, v64, causal)
    out, lse = _gpu_fwd(qkv, P, block, layout, causal, n_split=n_split)
    eo, el = _errs(out, lse, o_ref, l_ref)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)


def test_fwd_tiny_workload():
    w = WORKLOADS["tiny"]
    qkv, (q64, k64, v64) = _case(w["batch"], w["seq_len"], w["heads"], w["head_dim"],
                                 SEEDS["tiny"])
    o_ref, l_ref = oracle.attention_fwd(q64, k64, v64, w["causal"])
    for layout in ("contiguous", "striped"):
        for n_split in (1, 0):
            out, lse = _gpu_fwd(qkv, w["P"], w["block"], layout, w["causal"], n_split=n_split)
            eo, el = _errs(out, lse, o_ref, l_ref)
            assert eo <= OUT_TOL and el <= LSE_TOL, (layout, n_split, eo, el)


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_fwd_8k_workload(layout):
    w = WORKLOADS["8k"]
    qkv, (q64, k64, v64) = _case(w["batch"], w["seq_len"], w["heads"], w["head_dim"], SEEDS["8k"])
    o_ref, l_ref = oracle.attention_fwd(q64, k64, v64, True)
    out, lse, sw = _gpu_fwd(qkv, w["P"], w["block"], layout, True, shard_work=True)
    eo, el = _errs(out, lse, o_ref, l_ref)
    assert eo <= OUT_TOL and el <= LSE_TOL, (eo, el)
    # bf16 output: same bound plus bf16's own rounding of the exact value
    ob, _ = _gpu_fwd(qkv, w["P"], w["block"], layout, True, out_dtype=torch.bfloat16)
    diff = np.abs(ob.float().cpu().numpy() - o_ref)
    assert np.all(diff <= OUT_TOL + 2.0 ** -8 * np.abs(o_ref))
    # per-shard work: device counters == host closed form; striped, zigzag are balanced
    model = era.ra_shard_work_model(w["seq_len"], w["P"], w["block"], layout, True)
    got = sw.cpu().numpy().astype(np.int64)
    H = w["heads"]
    for u, name in enumerate(("tiles", "pairs", "visits")):
        assert list(got[u]) == [H * x for x in model[name]], name
    pairs = got[1].astype(np.float64)
    ratio = pairs.max() / pairs.mean()
    if layout != "contiguous":
        assert ratio <= 1.05
    else:
        assert ratio > 1.5


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_first_causal_token_is_exact(layout):
    qkv, (q64, k64, v64) = _case(2, 1024, 2, 128, seed=5)
    out, lse = _gpu_fwd(qkv, 4, 128, layout, True)
    o = out.cpu().numpy()
    assert np.array_equal(o[:, 0], v64[:, 0])
    s00 = np.einsum("bhd,bhd->bh", q64[:, 0], k64[:, 0]) / math.sqrt(128)
    assert np.max(np.abs(lse.cpu().numpy()[:, :, 0] - s00)) < 1e-5


def test_constant_v_gives_constant_output():
    q, k, _ = make_inputs(1, 2048, 2, 128, seed=6, with_dout=False)
    v = torch.linspace(-2, 3, 128).to(torch.bfloat16).expand(1, 2048, 2, 128).contiguous()
    for layout in ("contiguous", "striped", "zigzag"):
        out, _ = _gpu_fwd((q, k, v), 8, 128, layout, True)
        assert float((out.cpu() - v.float()).abs().max()) <= OUT_TOL


def test_layouts_agree_and_runs_are_deterministic():
    qkv, _ = _case(1, 4096, 4, 128, seed=9)
    oc, lc = _gpu_fwd(qkv, 8, 128, "contiguous", True)
    os_, ls = _gpu_fwd(qkv, 8, 128, "striped", True)
    assert float((oc - os_).abs().max()) <= OUT_TOL
    assert float((lc - ls).abs().max()) <= LSE_TOL
    os2, ls2 = _gpu_fwd(qkv, 8, 128, "striped", True)
    assert torch.equal(os_, os2) and torch.equal(ls, ls2)
    oz, lz = _gpu_fwd(qkv, 4, 128, "zigzag", True)
    assert float((oz - os_).abs().max()) <= OUT_TOL
    assert float((lz - ls).abs().max()) <= LSE_TOL


@pytest.mark.parametrize("n,D,B,L,H", [(3, 128, 1, 256, 2), (6, 128, 1, 256, 2), (1, 64, 1, 256, 2),
                                       (5, 24, 1, 256, 2), (2, 256, 1, 256, 2),
                                       (7, 128, 2, 384, 3), (4, 64, 3, 200, 5)])
def test_merge_entry_point_matches_oracle_merge(n, D, B, L, H):
    rng = np.random.default_rng(3 + n + D)
    o = rng.standard_normal((n, B, L, H, D)).astype(np.float32)
    lse = rng.standard_normal((n, B, H, L)).astype(np.float32)
    lse[n - 1, 0, 0, :7] = -np.inf
    o[n - 1, 0, :7, 0, :] = np.nan                  # a skipped partial's contents never matter
    lse[0, B - 1, H - 1, L - 3:] = -np.inf          # skipped in the first part, at the tail
    o[0, B - 1, L - 3:, H - 1, :] = np.nan
    lse[:, 0, 1, 5] = -np.inf                       # a row with no visible key at all
    o_or = np.where(np.isnan(o), 0.0, o).astype(np.float64)
    mo, ml = oracle.merge_partials(o_or, lse.astype(np.float64))
    go, gl = era.ra_merge(torch.from_numpy(o).cuda(), torch.from_numpy(lse).cuda(),
                          out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.max(np.abs(go.cpu().numpy() - mo)) < 1e-5
    gln = gl.cpu().numpy()
    assert gln[0, 1, 5] == -np.inf and np.all(go.cpu().numpy()[0, 5, 1] == 0)
    fin = np.isfinite(ml)
    assert np.max(np.abs(gln[fin] - ml[fin])) < 1e-5


def test_timeout_selftest_reports_and_recovers():
    ws = era.Workspace("cuda")
    era.ra_selftest_timeout(ws, timeout_us=2000)
    with pytest.raises(era.RaError, match="RA_ERR_DEVICE_TIMEOUT"):
        ws.check()
    ws.check()                                      # word cleared, context still usable
    qkv, _ = _case(1, 1024, 1, 128, seed=1)
    q, k, v = (t.cuda() for t in qkv)
    era.ra_fwd(q, k, v, 4, 128, "striped", True, workspace=ws)
    ws.check()
