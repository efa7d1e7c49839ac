"""NaN and Inf inputs on the GPU: they propagate where the fp64 oracle puts them, every
other output is unchanged, and no kernel waits in vain.

labhub "Ring Attention 論文分析", section "限界、失敗事例、そして未解決の問題" (the failure
case "NaN/Inf の発散"), names NaN/Inf from the online softmax as a hazard of the method.
A NaN in one element of q (row r) and, separately, +inf in one element of v (key c) are
planted on the host; ra_fwd and ra_bwd then run on the
poisoned inputs in every layout, with the ring steps fused (one online state) and split
(partials merged), and

* the workspace error word reports no timeout;
* the non-finite outputs (out, lse, dQ, dK, dV) are exactly the oracle's, element by element;
* the finite outputs match the oracle within the usual tolerances and equal those of a
  clean run (bit for bit where the kernels are deterministic: the forward, dK and dV; dQ
  within 1e-2 relative, its fp32 reductions land in any order).

Positions: r is the last row of a 128-row query tile and c the first key of a 128-key tile
(of shard 0 when striped) in every layout, and both sit at a 256-row block edge of the
oracle.  There, neither side has a masked (zero-probability) term beside the poisoned value
in a product: the kernels multiply masked probabilities as zeros, so elsewhere 0 * inf or
0 * NaN would spread a NaN across the rest of that tile.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300.synthetic import make_inputs, to_f64

pytestmark = pytest.mark.gpu

B, L, H, D, P, BLOCK = 1, 2048, 2, 128, 4, 128
R_NAN = 2 * 128 * P - 1        # last row of a query tile in every layout
C_INF = 128 * P                # first key of a KV tile in every layout (shard 0 if striped)
HP = 1                         # the poisoned head


def _run(q, k, v, do, layout, n_split, ws):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o32, l32 = era.ra_fwd(qd, kd, vd, P, BLOCK, layout, True, out_dtype=torch.float32,
                          n_split=n_split, workspace=ws)
    out, lse = era.ra_fwd(qd, kd, vd, P, BLOCK, layout, True, n_split=n_split, workspace=ws)
    dq, dk, dv = era.ra_bwd(qd, kd, vd, out, lse, dod, P, BLOCK, layout, True, workspace=ws)
    ws.check()                  # raises on a device timeout
    return {n: t.cpu() for n, t in
            (("out", o32), ("lse", l32), ("dq", dq), ("dk", dk), ("dv", dv))}


def _np(t):
    return t.double().numpy()


@pytest.mark.parametrize("poison", ["nan_q", "inf_v"])
@pytest.mark.parametrize("n_split", [1, 0])
@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_nonfinite_inputs_propagate_exactly(layout, n_split, poison):
    q, k, v, do = make_inputs(B, L, H, D, seed=91)
    qp, vp = q.clone(), v.clone()
    if poison == "nan_q":
        qp[0, R_NAN, HP, 3] = float("nan")
    else:
        vp[0, C_INF, HP, 5] = float("inf")
    ws = era.Workspace(torch.device("cuda:0"))
    got = _run(qp, k, vp, do, layout, n_split, ws)
    clean = _run(q, k, v, do, layout, n_split, ws)

    q64, k64, v64, do64 = to_f64(qp, k, vp, do)
    ro, rl = oracle.attention_fwd(q64, k64, v64, causal=True)
    rdq, rdk, rdv = oracle.attention_bwd(q64, k64, v64, do64, causal=True)
    ref = {"out": ro, "lse": rl, "dq": rdq, "dk": rdk, "dv": rdv}

    for name in ("out", "lse", "dq", "dk", "dv"):
        g, r, c = _np(got[name]), ref[name], _np(clean[name])
        fin = np.isfinite(r)
        assert np.array_equal(np.isfinite(g), fin), name
        assert (~fin).any() or name in ("lse", "dv"), name     # the poison reached it
        if name == "out":
            assert np.max(np.abs(g[fin] - r[fin])) <= 1e-2
        elif name == "lse":
            assert np.max(np.abs(g[fin] - r[fin])) <= 1e-3
        else:
            assert np.linalg.norm(g[fin] - r[fin]) / np.linalg.norm(r[fin]) <= 2e-2, name
        # the finite outputs are the clean run's
        if name == "dq":
            assert np.linalg.norm(g[fin] - c[fin]) / np.linalg.norm(c[fin]) <= 1e-2
        else:
            assert np.array_equal(g[fin], c[fin]), name
