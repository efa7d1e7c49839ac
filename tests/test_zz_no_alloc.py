"""ra_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such a caller (a plugin that receives tensors and a stream from a host runtime but no
allocator, or a latency-critical path that may not call cudaMalloc because it can stall
the device) has no workspace to pass; the entry point uses scratch memory built into the
library instead.  These tests call it through the C ABI and compare it with ra_bwd on the
same inputs, twice in a row, because the built-in scratch keeps the previous call's
contents, and once with the fp64 oracle.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300 import api
from exact_blockwise_ring_gb300.synthetic import make_inputs, to_f64

pytestmark = pytest.mark.gpu

GRAD_TOL = 2e-2


def _noalloc():
    f = api.lib().ra_bwd_noalloc
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(api.Params), P, P, P, P, ctypes.c_int, P, P, P, P, P, P]
    return f


def _rel(a, b):
    a, b = a.float(), b.float()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("layout,Hkv", [("striped", 4), ("zigzag", 2)])
def test_noalloc_backward_matches_workspace_backward_twice(layout, Hkv):
    torch.cuda.init()
    B, L, H, D, P, block = 1, 2048, 4, 128, 4, 128
    q, k, v, do = (t.cuda() for t in make_inputs(B, L, H, D, seed=77, kv_heads=Hkv))
    out, lse = era.ra_fwd(q, k, v, P, block, layout, True)
    ref = era.ra_bwd(q, k, v, out, lse, do, P, block, layout, True)
    torch.cuda.synchronize()
    f = _noalloc()
    prm = api.make_params(B, L, H, D, P, block, layout, True, kv_heads=Hkv)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        # poison the outputs so a call that wrote nothing cannot pass
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        st = f(ctypes.byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), 0,
               lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), stream)
        assert st == 0, api.lib().ra_last_error_message()
        torch.cuda.synchronize()
        for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            assert torch.isfinite(got).all(), (call, name)
            assert _rel(got, want) <= GRAD_TOL, (call, name, _rel(got, want))
        # dK and dV are accumulated on chip in a fixed order: the same bits as ra_bwd's
        # (dQ's fp32 reductions land in any order, so it is held to the tolerance above)
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), call
    # and against the fp64 oracle (grouped-query backward on the same bf16 inputs)
    g_ref = oracle.gqa_bwd(*to_f64(q, k, v, do), causal=True)
    for got, want, name in zip((dq, dk, dv), g_ref, ("dq", "dk", "dv")):
        e = float(np.linalg.norm(got.double().cpu().numpy() - want) / np.linalg.norm(want))
        assert e <= GRAD_TOL, (name, e)


def test_noalloc_rejects_problems_beyond_its_scratch():
    f = _noalloc()
    # 32768 tokens x 32 heads x 128 needs ~520 MiB of scratch: far above the built-in 64 MiB
    prm = api.make_params(1, 32768, 32, 128, 8, 128, "striped", True)
    fake = ctypes.c_void_p(1 << 20)
    st = f(ctypes.byref(prm), fake, fake, fake, fake, 0, fake, fake, fake, fake, fake, None)
    assert st == 3
    assert "scratch" in api.lib().ra_last_error_message().decode()
