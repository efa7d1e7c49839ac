"""Sweep of every kernel through the checked build of the library (run by
test_gpu_checked.py in a child process with RA_LIBRARY pointing at libra_checked.so).

Each kernel range-checks its TMA box coordinates, TMEM columns and lane quarters,
shared-memory operand offsets, global element indices and per-role item counts; a
violation would make ra_check_error() report RA_ERR_CHECK.  The sweep covers the forward
(fused and split, every layout, causal and not, P from 1 to 8, blocks 128 and 256, head dims
64 and 128, grouped-query heads), the backward on the same grid, the merge, and one small
blockwise transformer layer forward and backward; a few cases are also compared with the
fp64 oracle.  Prints CHECKED SWEEP OK at the end.
"""

import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle                                           # noqa: E402
import exact_blockwise_ring_gb300 as era                # noqa: E402
from exact_blockwise_ring_gb300 import api              # noqa: E402
from exact_blockwise_ring_gb300.synthetic import make_bpt_weights, make_inputs, to_f64  # noqa: E402

CASES = [
    # B, L, H, Hkv, D, P, block, layout, causal, n_split
    (1, 1024, 2, 2, 128, 4, 128, "contiguous", True, 1),
    (1, 1024, 2, 2, 128, 4, 128, "striped", True, 0),
    (2, 2048, 3, 3, 128, 2, 128, "zigzag", True, 1),
    (1, 1536, 2, 2, 128, 4, 128, "striped", True, 2),
    (1, 2048, 2, 2, 128, 4, 256, "zigzag", True, 0),
    (1, 1024, 1, 1, 128, 1, 128, "contiguous", True, 1),
    (1, 1024, 2, 2, 128, 8, 128, "striped", True, 1),
    (1, 1024, 2, 2, 128, 4, 128, "striped", False, 1),
    (1, 1024, 2, 2, 64, 4, 128, "zigzag", True, 0),
    (1, 2048, 4, 2, 128, 4, 128, "striped", True, 1),
    (1, 2048, 4, 1, 64, 2, 256, "contiguous", True, 2),
]


def main():
    assert api.lib().ra_checks_enabled() == 1, "not the checked build: %s" % api.LIB_PATH
    dev = torch.device("cuda:0")
    ws = era.Workspace(dev)
    for n, (B, L, H, Hkv, D, P, blk, layout, causal, n_split) in enumerate(CASES):
        q, k, v, do = make_inputs(B, L, H, D, seed=500 + n, kv_heads=Hkv)
        qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
        out, lse, sw = era.ra_fwd(qd, kd, vd, P, blk, layout, causal, n_split=n_split,
                                  shard_work=True, workspace=ws)
        ws.check()
        dq, dk, dv = era.ra_bwd(qd, kd, vd, out, lse, dod, P, blk, layout, causal, workspace=ws)
        ws.check()
        if n % 3 == 0:       # a few against the oracle as well
            q64, k64, v64, do64 = to_f64(q, k, v, do)
            ro, rl = oracle.gqa_fwd(q64, k64, v64, causal)
            rg = oracle.gqa_bwd(q64, k64, v64, do64, causal)
            o = out.double().cpu().numpy()
            assert np.max(np.abs(o - ro)) <= 1e-2 + 2.0 ** -8 * np.max(np.abs(ro)), n
            assert np.max(np.abs(lse.double().cpu().numpy() - rl)) <= 1e-3, n
            for g, r in zip((dq, dk, dv), rg):
                assert np.linalg.norm(g.double().cpu().numpy() - r) / np.linalg.norm(r) <= 2e-2
        print("case", n, "ok", flush=True)
    # the merge on its own
    o_parts = torch.randn((3, 1, 512, 2, 128), device=dev)
    lse_parts = torch.randn((3, 1, 2, 512), device=dev)
    era.ra_merge(o_parts, lse_parts)
    ws.check()
    # one small blockwise transformer layer, forward and backward (GEMMs, LayerNorms)
    d, d_ff, L = 512, 1024, 1024
    x = make_inputs(1, L, 1, d, seed=601, with_dout=False)[0].view(1, L, d).to(dev)
    w = {name: t.to(dev) for name, t in make_bpt_weights(d, d_ff, seed=602).items()}
    era.ra_bpt_fwd(x, w, 4, 4, 128, "zigzag", True, block_rows=256, workspace=ws, train=True)
    ws.check()
    dy = make_inputs(1, L, 1, d, seed=603, with_dout=False)[0].view(1, L, d).to(dev)
    era.ra_bpt_bwd(x, w, dy, 4, 4, 128, "zigzag", True, block_rows=256, workspace=ws)
    ws.check()
    torch.cuda.synchronize()
    print("CHECKED SWEEP OK", flush=True)


if __name__ == "__main__":
    main()
