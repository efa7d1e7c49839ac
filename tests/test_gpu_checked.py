"""The checked build (libra_checked.so: every kernel range-checks its indices and item
counts before use) over a sweep of every kernel, in a child process that loads it through
RA_LIBRARY.  It stands in for a memory checker: a range violation is reported through the
workspace error word (RA_ERR_CHECK) instead of an out-of-range access."""

import os
import subprocess
import sys

import pytest

from exact_blockwise_ring_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checked_lib():
    return build.build(checked=True)


def test_checked_build_sweep(checked_lib):
    env = dict(os.environ, RA_LIBRARY=checked_lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_sweep.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "CHECKED SWEEP OK" in r.stdout


def test_normal_build_reports_no_checks():
    from exact_blockwise_ring_gb300 import api
    if os.environ.get("RA_LIBRARY"):
        pytest.skip("RA_LIBRARY selects another build")
    assert api.lib().ra_checks_enabled() == 0
