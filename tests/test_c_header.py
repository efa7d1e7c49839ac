"""The boundary is a C ABI: include/ra.h must compile as strict C99, the ctypes mirrors in
the binding must have the same struct sizes, field offsets and enum values as the header,
and a plain C program must be able to link the library and call it.  Host-only (the calls
made here never reach CUDA)."""

import ctypes
import os
import shutil
import subprocess

import pytest

from exact_blockwise_ring_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")

STRUCTS = {"ra_params_t": api.Params, "ra_bpt_params_t": api.BptParams,
           "ra_bpt_weights_t": api.BptWeights, "ra_bpt_grads_t": api.BptGrads}

ENUMS = {"RA_OK": 0, "RA_ERR_INVALID_ARG": 1, "RA_ERR_UNSUPPORTED": 2, "RA_ERR_WORKSPACE": 3,
         "RA_ERR_CUDA": 4, "RA_ERR_DEVICE_TIMEOUT": 5, "RA_ERR_CHECK": 6, "RA_LAYOUT_CONTIGUOUS": 0,
         "RA_LAYOUT_STRIPED": 1, "RA_LAYOUT_ZIGZAG": 2, "RA_BF16": api.RA_BF16,
         "RA_FP32": api.RA_FP32, "RA_EPI_BIAS": api.EPILOGUES["bias"],
         "RA_EPI_BIAS_GELU": api.EPILOGUES["bias_gelu"],
         "RA_EPI_BIAS_RESIDUAL": api.EPILOGUES["bias_residual"]}


def _compile_and_run(tmp_path, body, link=False):
    src = tmp_path / "client.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "ra.h"\n'
                   "int main(void) {\n" + body + "  return 0;\n}\n")
    exe = tmp_path / "client"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", INCLUDE,
           str(src), "-o", str(exe)]
    if link:
        libdir = os.path.dirname(api.LIB_PATH)
        cmd += ["-L", libdir, "-l:libra.so", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    return r.stdout.split("\n")


def test_header_layout_matches_the_binding(tmp_path):
    body = ""
    for cname, cls in STRUCTS.items():
        body += '  printf("%s size %%zu\\n", sizeof(%s));\n' % (cname, cname)
        for f, _ in cls._fields_:
            body += '  printf("%s.%s %%zu\\n", offsetof(%s, %s));\n' % (cname, f, cname, f)
    for e in ENUMS:
        body += '  printf("%s %%d\\n", (int)%s);\n' % (e, e)
    got = dict(line.rsplit(" ", 1) for line in _compile_and_run(tmp_path, body) if line)
    for cname, cls in STRUCTS.items():
        assert int(got[cname + " size"]) == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert int(got["%s.%s" % (cname, f)]) == getattr(cls, f).offset, (cname, f)
    for e, v in ENUMS.items():
        assert int(got[e]) == v, e


@pytest.fixture(scope="module")
def built():
    if not os.path.exists(api.LIB_PATH):
        from exact_blockwise_ring_gb300 import build
        build.build()
    return api.LIB_PATH


def test_c_client_links_and_calls_the_library(tmp_path, built):
    # the zigzag work model of a 4-shard causal ring, and a rejected layer shape, from C
    body = r"""
  ra_params_t p = {1, 4096, 2, 128, 128, 4, RA_LAYOUT_ZIGZAG, 1, 0.0f, 0, 0};
  unsigned long long w[12];
  ra_bpt_params_t b = {{1, 1024, 2, 128, 128, 4, RA_LAYOUT_STRIPED, 1, 0.0f, 0, 0}, 1024, 256, 0.0f};
  ra_status_t s = ra_shard_work_model(&p, w);
  int i;
  printf("status %s\n", ra_status_string(s));
  for (i = 0; i < 12; ++i) printf("w%d %llu\n", i, w[i]);
  printf("bpt_ws %zu\n", ra_bpt_workspace_bytes(&b));
  s = ra_bpt_fwd(&b, NULL, NULL, NULL, RA_BF16, NULL, 0, NULL);
  printf("bpt_status %d\n", (int)s);
  printf("bpt_msg %s\n", ra_last_error_message());
"""
    lines = [x for x in _compile_and_run(tmp_path, body, link=True) if x]
    kv = dict(x.split(" ", 1) for x in lines)
    assert kv["status"] == "RA_OK"
    want = api.ra_shard_work_model(4096, 4, 128, "zigzag", True)
    flat = want["tiles"] + want["pairs"] + want["visits"]
    assert [int(kv["w%d" % i]) for i in range(12)] == flat
    assert len(set(want["pairs"])) == 1          # zigzag: equal work on every shard
    assert kv["bpt_ws"] == "0"                   # d_model 256 is not a multiple of 512
    assert int(kv["bpt_status"]) == 2 and "multiple of 512" in kv["bpt_msg"]
