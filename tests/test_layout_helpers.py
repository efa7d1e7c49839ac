"""The token-assignment and ring-schedule helpers the kernels share (csrc/ra_internal.h:
token_of, shard_local_of, tokens_upto, RingSched's q_end / q_diag / u_end for the forward
and BwdSched's t_lo / delta for the backward), compiled for
the host and checked against brute force built on the oracle's token assignment
(oracle/work.py) over a seeded sweep of small shapes, every layout, causal or not.

RingSched is checked as the forward kernel uses it (units of two query tiles, t0 = 2s): the
KV tiles of shard j that query tile t sees must be a prefix of length q_end, every tile of
it but a masked diagonal must be fully visible, and q_diag must name that diagonal (the
pages' rule, labhub section "Causal Masking の処理": later blocks skipped, the same block
masked, earlier ones full, decided here from original token positions)."""

import os
import random
import shutil
import subprocess

import pytest

import oracle
from oracle.work import shard_of, local_of, shard_tokens, tile_class

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"
LAYOUTS = {"contiguous": 0, "striped": 1, "zigzag": 2}

pytestmark = pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC),
                                reason="needs g++ and the CUDA headers")

HARNESS = r"""
#include <cstdio>
#include <cstdlib>
#include "ra_internal.h"
using namespace ra;
int main(int argc, char** argv) {
  if (argc < 6) return 2;
  const int layout = atoi(argv[1]), P = atoi(argv[2]);
  const long long n = atoll(argv[3]);
  const int T = atoi(argv[4]), causal = atoi(argv[5]);
  if (argc > 6) {   // the backward's schedule (128-row tiles): t_lo, then delta per tile
    printf("B");
    for (int j = 0; j < P; ++j)
      for (int u = 0; u < T; ++u) {
        const BwdSched sc{j, u, (int)n, T, P, layout, causal};
        for (int k = 0; k < P; ++k) {
          const int i = sc.i_of(k);
          printf(" %d %d", i, sc.t_lo(i));
          for (int t = 0; t < T; ++t) printf(" %lld", sc.delta(i, t));
        }
      }
    printf("\n");
    return 0;
  }
  printf("T");
  for (int i = 0; i < P; ++i)
    for (long long a = 0; a < n; ++a) printf(" %lld", token_of(layout, i, a, n, P));
  printf("\nS");
  for (long long tok = 0; tok < P * n; ++tok) {
    long long s, l;
    shard_local_of(layout, tok, n, P, &s, &l);
    printf(" %lld %lld", s, l);
  }
  printf("\nU");
  for (int j = 0; j < P; ++j)
    for (long long tok = -1; tok <= P * n; ++tok) printf(" %lld", tokens_upto(layout, j, tok, n, P));
  printf("\nQ");
  for (int i = 0; i < P; ++i)
    for (int s = 0; 2 * s < T; ++s) {
      const RingSched sc{i, 2 * s, 2, T, P, layout, causal, 0, P};
      for (int j = 0; j < P; ++j)
        printf(" %d %d %d %d %d", sc.q_end(0, j), sc.q_end(1, j), sc.q_diag(0, j), sc.q_diag(1, j),
               sc.u_end(j));
    }
  printf("\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    d = tmp_path_factory.mktemp("layout_helpers")
    src = d / "harness.cpp"
    src.write_text(HARNESS)
    exe = d / "harness"
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-I", CUDA_INC, "-I",
                        os.path.join(ROOT, "exact_blockwise_ring_gb300", "csrc"), "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(exe)


def _run(exe, layout, P, n, T, causal):
    out = subprocess.run([exe, str(LAYOUTS[layout]), str(P), str(n), str(T), str(int(causal))],
                         capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    rows = {}
    for ln in out.stdout.splitlines():
        f = ln.split()
        rows[f[0]] = [int(x) for x in f[1:]]
    return rows


def _ring_ref(tokens, i, j, t, T, bt, causal):
    """(q_end, q_diag) of query tile t of shard i against KV shard j, by brute force."""
    if t >= T:
        return 0, -1
    q = tokens[i][t * bt:(t + 1) * bt]
    cls = [tile_class(q, tokens[j][u * bt:(u + 1) * bt], causal) for u in range(T)]
    vis = [c != "skip" for c in cls]
    e = sum(vis)
    assert vis == [True] * e + [False] * (T - e), "visible KV tiles are not a prefix"
    diags = [u for u, c in enumerate(cls) if c == "diag"]
    assert len(diags) <= 1 and all(c == "full" for c in cls[:e - len(diags)])
    if diags:
        assert diags[0] == e - 1, "the masked tile is not the last visible one"
    return e, (diags[0] if diags else -1)


def test_layout_helpers_match_brute_force(harness):
    rng = random.Random(1202)
    for _ in range(120):
        layout = rng.choice(list(LAYOUTS))
        causal = rng.random() < 0.85
        P = rng.randint(1, 7)
        T = rng.randint(1, 5) * (2 if layout == "zigzag" else 1)
        bt = rng.randint(2, 5)                    # tokens per tile (the kernels use 128)
        n = T * bt
        L = P * n
        got = _run(harness, layout, P, n, T, causal)
        tokens = [shard_tokens(i, L, P, layout) for i in range(P)]
        assert got["T"] == [tok for i in range(P) for tok in tokens[i]]
        assert got["S"] == [v for tok in range(L)
                            for v in (shard_of(tok, L, P, layout), local_of(tok, L, P, layout))]
        assert got["U"] == [sum(1 for x in tokens[j] if x <= tok)
                            for j in range(P) for tok in range(-1, L + 1)]
        want_q = []
        for i in range(P):
            for s in range(0, (T + 1) // 2):
                for j in range(P):
                    e0, d0 = _ring_ref(tokens, i, j, 2 * s, T, bt, causal)
                    e1, d1 = _ring_ref(tokens, i, j, 2 * s + 1, T, bt, causal)
                    want_q += [e0, e1, d0, d1, max(e0, e1)]
        assert got["Q"] == want_q, (layout, P, T, bt, causal)


def test_backward_schedule_matches_brute_force(harness):
    # BwdSched with the kernels' 128-row tiles: the query shards come in ring order, the
    # visible query tiles of a shard are a suffix t >= t_lo, and inside a tile pair key row
    # b is visible to query row a exactly when a - b + delta >= 0
    rows = [0, 1, 2, 63, 64, 65, 126, 127]
    rng = random.Random(77)
    for _ in range(24):
        layout = rng.choice(list(LAYOUTS))
        causal = rng.random() < 0.8
        P = rng.randint(1, 5)
        T = rng.randint(1, 3) * (2 if layout == "zigzag" else 1)
        n = 128 * T
        L = P * n
        out = subprocess.run([harness, str(LAYOUTS[layout]), str(P), str(n), str(T),
                              str(int(causal)), "bwd"], capture_output=True, text=True, timeout=60)
        assert out.returncode == 0, out.stderr
        vals = [int(x) for x in out.stdout.split()[1:]]
        tokens = [shard_tokens(i, L, P, layout) for i in range(P)]
        pos = 0
        for j in range(P):
            for u in range(T):
                kt = tokens[j][u * 128:(u + 1) * 128]
                for i in [(j + k) % P for k in range(P)]:     # i = (j + k) mod P
                    gi, t_lo = vals[pos], vals[pos + 1]
                    deltas = vals[pos + 2:pos + 2 + T]
                    pos += 2 + T
                    assert gi == i
                    vis = [min(kt) <= max(tokens[i][t * 128:(t + 1) * 128]) if causal else True
                           for t in range(T)]
                    want_lo = vis.index(True) if True in vis else T
                    assert vis == [False] * want_lo + [True] * (T - want_lo)
                    assert t_lo == want_lo, (layout, P, T, j, u, i)
                    if causal:
                        for t in range(T):
                            qt = tokens[i][t * 128:(t + 1) * 128]
                            for a in rows:
                                for b in rows:
                                    assert (a - b + deltas[t] >= 0) == (kt[b] <= qt[a])
        assert pos == len(vals)


def test_planted_schedule_error_is_caught():
    # the brute force is not vacuous: a schedule that drops the diagonal tile, or takes a
    # striped KV shard after the query shard as fully visible, disagrees with it
    L, P, bt, T = 24, 3, 2, 4
    tokens = [shard_tokens(i, L, P, "striped") for i in range(P)]
    e, d = _ring_ref(tokens, 0, 2, 1, T, bt, True)
    assert (e, d) == (2, 1)
    q = tokens[0][2:4]
    assert tile_class(q, tokens[2][2:4], True) == "diag"      # not "full": j > i masks b = a
    assert oracle.ring_order(0, P) == [0, 2, 1]


UMAX_HARNESS = r"""
#include <cstdio>
#include "ra_internal.h"
using namespace ra;
int main() {
  // u_max of a striped unit (query tiles 4 and 5) over every ring step: its longest prefix
  const RingSched sc{1, 4, 2, 9, 4, RA_LAYOUT_STRIPED, 1, 0, 4};
  // and of a contiguous unit of shard 1 (tiles 4, 5 of 9): every KV tile of shard 0
  const RingSched sd{1, 4, 2, 9, 4, RA_LAYOUT_CONTIGUOUS, 1, 0, 4};
  printf("U %d %d\n", sc.u_max(), sd.u_max());
  return 0;
}
"""


def test_u_max(tmp_path):
    """u_max, the tile-outer walk's bound: the longest visible KV-tile prefix of a unit over
    its ring steps."""
    src = tmp_path / "umax.cpp"
    src.write_text(UMAX_HARNESS)
    exe = tmp_path / "umax"
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-I", CUDA_INC, "-I",
                        os.path.join(ROOT, "exact_blockwise_ring_gb300", "csrc"), "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60).stdout
    assert "U 6 9" in out
