"""Build libra.so in-tree: every CUDA source under csrc/ for sm_103a, in parallel.

Run ``python -m exact_blockwise_ring_gb300.build`` (or ``__graft_entry__.build()``).
Object files go to ``_build/`` next to this file; the shared library to this folder.

``build(checked=True)`` (``python -m exact_blockwise_ring_gb300.build --checked``) builds
the checked variant libra_checked.so (objects in ``_build_checked/``): the same sources
compiled with RA_CHECKS, so that every kernel range-checks its indices before use and
reports a violation through the workspace error word (ra_check_error: RA_ERR_CHECK)
instead of touching memory out of range.  Select it at run time with RA_LIBRARY.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libra.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "libra_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I" + os.path.join(HERE, "..", "include")]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")
    return cand


def _compile(nvcc, src, obj, extra=()):
    cmd = [nvcc] + ARCH + FLAGS + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
    return obj


def build(verbose=False, checked=False):
    """Compile csrc/*.cu and link libra.so (libra_checked.so with checked=True). Returns
    the library path."""
    nvcc = _nvcc()
    bdir = BUILD_CHECKED if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    extra = ["-DRA_CHECKS"] if checked else []
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        for f in srcs:
            obj = os.path.join(bdir, f[:-3] + ".o")
            jobs.append(ex.submit(_compile, nvcc, os.path.join(CSRC, f), obj, extra))
        objs = [j.result() for j in jobs]
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib


if __name__ == "__main__":
    build(verbose=True, checked="--checked" in sys.argv)
    sys.exit(0)
