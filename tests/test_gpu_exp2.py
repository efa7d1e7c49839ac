"""The two 2^x forms the softmax kernels mix, on the GPU through ra_selftest_exp2: the
software form (range reduction and a polynomial on the FMA pipe) against exact 2^x within
its derived relative error bound over the whole input range the kernels use, against the
hardware unit's ex2.approx.ftz, and at the special values (-inf and x <= -127 give 0, NaN
gives NaN, integers give exact powers of two)."""

import numpy as np
import pytest
import torch

import exact_blockwise_ring_gb300 as era

pytestmark = pytest.mark.gpu

SOFT_BOUND = 4e-6          # the polynomial's 3.6e-6 plus float32 evaluation
HW_BOUND = 2.0 ** -21      # ex2.approx.ftz: a few ulp (measured, not a derived bound)


def test_software_exp2_matches_exact_and_hardware():
    xs = np.concatenate([np.linspace(-126.0, 8.0, 1_000_003), np.arange(-126, 9, dtype=np.float64),
                         np.arange(-126, 8) + 0.5, np.linspace(-1, 1, 100_001)])
    x = torch.tensor(xs, dtype=torch.float32)
    soft, hw = era.ra_selftest_exp2(x.cuda())
    torch.cuda.synchronize()
    x64 = x.double().numpy()
    want = np.exp2(x64)
    s = soft.double().cpu().numpy()
    h = hw.double().cpu().numpy()
    normal = want >= 2.0 ** -126
    assert np.max(np.abs(s[normal] / want[normal] - 1)) < SOFT_BOUND
    assert np.max(np.abs(h[normal] / want[normal] - 1)) < HW_BOUND
    ints = x64 == np.round(x64)
    assert np.array_equal(s[ints & normal], want[ints & normal])      # 2^n exactly


def test_software_exp2_special_values():
    x = torch.tensor([-float("inf"), -1e30, -200.0, -127.0, -126.6, float("nan"), 0.0, -0.0,
                      1.0, 7.5], dtype=torch.float32)
    soft, hw = era.ra_selftest_exp2(x.cuda())
    torch.cuda.synchronize()
    s = soft.cpu().numpy()
    assert np.all(s[:5] == 0.0) and not np.signbit(s[:5]).any()       # +0 below the range
    assert np.isnan(s[5]) and np.isnan(hw.cpu().numpy()[5])
    assert s[6] == 1.0 and s[7] == 1.0 and s[8] == 2.0
    assert abs(s[9] / 2.0 ** 7.5 - 1) < SOFT_BOUND
