"""A failure already recorded in the workspace stops the later kernels of the path.

Every bounded wait in the kernels sets the workspace error word when it gives up; every
CTA launched after that reads the word at its start and leaves before it loads, waits
or allocates anything.  These tests plant the word on the host (the value a timeout
writes), run the forward, the backward and a layer GEMM on it, and check that each call
returns, that ra_check_error reports the word once and clears it, and that the next calls
compute the oracle's results: no GPU fault and no real timeout is involved.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300.synthetic import make_inputs, to_f64

pytestmark = pytest.mark.gpu

TIMEOUT_WORD = 0x7          # what a wait that gave up writes


def _plant(ws):
    # on the buffer the next calls will use: a workspace grows (into a fresh zeroed
    # buffer) on the first call that needs more, so the tests size it with a clean call
    ws.buf[:4].view(torch.int32).fill_(TIMEOUT_WORD)


@pytest.mark.parametrize("layout", ["striped", "zigzag"])
def test_attention_kernels_leave_at_once_after_a_recorded_failure(layout):
    q, k, v, do = make_inputs(1, 2048, 2, 128, seed=77)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    ws = era.Workspace(torch.device("cuda:0"))
    out, lse = era.ra_fwd(qd, kd, vd, 4, 128, layout, True, workspace=ws)
    era.ra_bwd(qd, kd, vd, out, lse, dod, 4, 128, layout, True, workspace=ws)
    ws.check()

    _plant(ws)
    out, lse = era.ra_fwd(qd, kd, vd, 4, 128, layout, True, workspace=ws)
    era.ra_bwd(qd, kd, vd, out, lse, dod, 4, 128, layout, True, workspace=ws)
    with pytest.raises(era.RaError, match="RA_ERR_DEVICE_TIMEOUT"):
        ws.check()
    ws.check()                               # reported once, then cleared

    out, lse = era.ra_fwd(qd, kd, vd, 4, 128, layout, True, workspace=ws)
    dq, dk, dv = era.ra_bwd(qd, kd, vd, out, lse, dod, 4, 128, layout, True, workspace=ws)
    ws.check()
    q64, k64, v64, do64 = to_f64(q, k, v, do)
    ro, rl = oracle.attention_fwd(q64, k64, v64, causal=True)
    assert np.max(np.abs(out.float().cpu().numpy() - ro)) <= 1.5e-2
    assert np.max(np.abs(lse.cpu().numpy() - rl)) <= 1e-3
    for g, r in zip((dq, dk, dv), oracle.attention_bwd(q64, k64, v64, do64, causal=True)):
        gn = g.double().cpu().numpy()
        assert np.linalg.norm(gn - r) / np.linalg.norm(r) <= 2e-2


def test_split_forward_and_merge_after_a_recorded_failure():
    q, k, v, _ = make_inputs(1, 1024, 2, 128, seed=78)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    ws = era.Workspace(torch.device("cuda:0"))
    era.ra_fwd(qd, kd, vd, 4, 128, "striped", True, n_split=0, workspace=ws)
    ws.check()
    _plant(ws)
    era.ra_fwd(qd, kd, vd, 4, 128, "striped", True, n_split=0, workspace=ws)
    with pytest.raises(era.RaError, match="RA_ERR_DEVICE_TIMEOUT"):
        ws.check()
    out, lse = era.ra_fwd(qd, kd, vd, 4, 128, "striped", True, n_split=0, workspace=ws,
                          out_dtype=torch.float32)
    ws.check()
    ro, rl = oracle.attention_fwd(*to_f64(q, k, v), causal=True)
    assert np.max(np.abs(out.cpu().numpy() - ro)) <= 1e-2
    assert np.max(np.abs(lse.cpu().numpy() - rl)) <= 1e-3


def test_layer_gemm_after_a_recorded_failure():
    g = torch.Generator().manual_seed(79)
    x = torch.randn(512, 256, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(512, 256, generator=g) / 16).to(torch.bfloat16).cuda()
    bias = torch.randn(512, generator=g).cuda()
    ws = era.Workspace(torch.device("cuda:0"))
    era.ra_linear(x, w, bias, "bias", workspace=ws)
    ws.check()
    _plant(ws)
    era.ra_linear(x, w, bias, "bias", workspace=ws)
    with pytest.raises(era.RaError, match="RA_ERR_DEVICE_TIMEOUT"):
        ws.check()
    y = era.ra_linear(x, w, bias, "bias", workspace=ws)
    ws.check()
    ref = x.double().cpu() @ w.double().cpu().T + bias.double().cpu()
    assert torch.max(torch.abs(y.double().cpu() - ref)) <= 0.05 * torch.max(torch.abs(ref))
