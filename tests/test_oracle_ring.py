"""Pins for the oracle's ring emulator, partial merge and work model (CPU only)."""

import os

import numpy as np
import pytest

import oracle
from oracle import work as owork

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(B, L, H, D, seed):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((B, L, H, D)) for _ in range(3))


# ---- the method reaches full attention exactly (up to rounding order) -----------

@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P,block", [(1, 8), (2, 4), (4, 2), (4, 8), (8, 4)])
def test_ring_equals_full_attention(layout, causal, P, block):
    L = 64
    q, k, v = _rand(1, L, 2, 8, seed=P * 10 + block)
    ro, rl = oracle.ring_fwd(q, k, v, P, layout, causal, block)
    fo, fl = oracle.attention_fwd(q, k, v, causal)
    assert np.max(np.abs(ro - fo)) < 1e-12
    assert np.max(np.abs(rl - fl)) < 1e-12


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("causal", [False, True])
def test_merged_partials_equal_full_attention(layout, causal):
    q, k, v = _rand(2, 32, 1, 4, seed=3)
    op, lp = oracle.ring_partials(q, k, v, 4, layout, causal, block=4)
    mo, ml = oracle.merge_partials(op, lp)
    fo, fl = oracle.attention_fwd(q, k, v, causal)
    assert np.max(np.abs(mo - fo)) < 1e-12
    assert np.max(np.abs(ml - fl)) < 1e-12


def test_striped_partials_have_fully_masked_rows():
    # striped, causal: at a step whose KV shard j is after the query shard i, the
    # query of local index 0 sees no key (its only candidate, key local 0 of shard j,
    # is a later token), so that partial has lse = -inf and O = 0.
    L, P = 32, 4
    q, k, v = _rand(1, L, 1, 4, seed=4)
    op, lp = oracle.ring_partials(q, k, v, P, "striped", True, block=4)
    for i in range(P):
        for kk in range(P):
            j = (i - kk) % P
            if j > i:
                assert lp[kk, 0, 0, i] == -np.inf
                assert np.all(op[kk, 0, i, 0, :] == 0)
    assert np.all(np.isfinite(lp[0]))          # step 0 (own shard): every row sees a key


def test_merge_single_partial_is_identity():
    q, k, v = _rand(1, 16, 1, 4, seed=5)
    fo, fl = oracle.attention_fwd(q, k, v, True)
    mo, ml = oracle.merge_partials(fo[None], fl[None])
    assert np.max(np.abs(mo - fo)) < 1e-15 and np.max(np.abs(ml - fl)) < 1e-15


def test_merge_closed_form_two_equal_partials():
    # two partials with equal lse and outputs O1, O2 merge to lse + ln 2 and (O1+O2)/2
    o = np.random.default_rng(6).standard_normal((2, 1, 8, 1, 4))
    l_ = np.full((2, 1, 1, 8), 0.3)
    mo, ml = oracle.merge_partials(o, l_)
    assert np.max(np.abs(ml - (0.3 + np.log(2.0)))) < 1e-15
    assert np.max(np.abs(mo - 0.5 * (o[0] + o[1]))) < 1e-15


@pytest.mark.parametrize("layout", ["striped", "zigzag"])
@pytest.mark.parametrize("causal", [False, True])
def test_permutation_equivariance(layout, causal):
    """Permute tokens into shard-major order, attend with the mask taken on original
    positions, unpermute: the output equals natural-order attention."""
    L, P = 48, 4
    q, k, v = _rand(1, L, 1, 8, seed=7)
    perm = np.concatenate([owork.shard_tokens(i, L, P, layout) for i in range(P)])
    qp, kp, vp = q[:, perm], k[:, perm], v[:, perm]
    s = (qp[0, :, 0] @ kp[0, :, 0].T) / np.sqrt(8)
    if causal:
        s = np.where(perm[None, :] > perm[:, None], -np.inf, s)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    op = p @ vp[0, :, 0]
    out = np.empty_like(op)
    out[perm] = op
    fo, _ = oracle.attention_fwd(q, k, v, causal)
    assert np.max(np.abs(out - fo[0, :, 0])) < 1e-13
    so, _ = oracle.ring_fwd(q, k, v, P, layout, causal, block=2)
    assert np.max(np.abs(so - fo)) < 1e-12


# ---- ring order and assignment ----------------------------------------------------

def test_ring_order_golden():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "ring_order.txt"))
            if ln.strip() and not ln.startswith("#")]
    for row in rows:
        P, dev = int(row[0]), int(row[1])
        order = oracle.ring_order(dev, P)
        for kk, want in enumerate(row[2:]):
            if want != "x":
                assert order[kk] == int(want), (dev, kk)


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_assignment_is_a_partition(layout):
    L, P = 96, 8
    seen = sorted(t for i in range(P) for t in oracle.shard_tokens(i, L, P, layout))
    assert seen == list(range(L))
    for t in range(L):
        i, a = oracle.shard_of(t, L, P, layout), oracle.local_of(t, L, P, layout)
        assert oracle.shard_tokens(i, L, P, layout)[a] == t


def test_zigzag_holds_symmetric_chunks():
    # L = 16, P = 4: chunks of 2; shard 1 holds chunk 1 (tokens 2, 3) and chunk 6 (12, 13)
    assert oracle.shard_tokens(1, 16, 4, "zigzag") == [2, 3, 12, 13]
    assert [oracle.shard_of(t, 16, 4, "zigzag") for t in range(16)] == \
        [0, 0, 1, 1, 2, 2, 3, 3, 3, 3, 2, 2, 1, 1, 0, 0]


def test_striped_is_round_robin():
    assert [oracle.shard_of(t, 32, 4, "striped") for t in range(8)] == [0, 1, 2, 3] * 2
    assert [oracle.shard_of(t, 32, 4, "contiguous") for t in (0, 7, 8, 31)] == [0, 0, 1, 3]


# ---- per-shard work model ---------------------------------------------------------

def _golden_demo():
    rows = {}
    for ln in open(os.path.join(GOLDEN, "work_demo.txt")):
        if ln.strip() and not ln.startswith("#"):
            f = ln.split()
            rows[f[0]] = ([int(x) for x in f[1:5]], float(f[5]), int(f[6]))
    return rows


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_work_model_reproduces_demo(layout):
    want, ratio, total = _golden_demo()[layout]
    w = oracle.shard_work(32, 4, 8, layout, causal=True)["visits"]
    assert w == want
    assert round(max(w) / min(w), 2) == ratio and sum(w) == total


@pytest.mark.parametrize("L,P,block", [(64, 4, 4), (256, 8, 8), (512, 4, 16), (128, 2, 64)])
def test_work_model_closed_forms(L, P, block):
    n = L // P
    T = n // block
    c = oracle.shard_work(L, P, block, "contiguous", causal=True)
    s = oracle.shard_work(L, P, block, "striped", causal=True)
    for i in range(P):
        assert c["tiles"][i] == i * T * T + T * (T + 1) // 2
        assert s["tiles"][i] == P * T * (T + 1) // 2
        assert c["pairs"][i] == n * (i * n) + n * (n + 1) // 2
        assert s["pairs"][i] == P * n * (n - 1) // 2 + n * (i + 1)
    assert sum(c["pairs"]) == sum(s["pairs"]) == L * (L + 1) // 2
    nc = oracle.shard_work(L, P, block, "striped", causal=False)
    assert nc["tiles"] == [P * T * T] * P and nc["pairs"] == [n * L] * P


@pytest.mark.parametrize("L,P,block", [(64, 4, 4), (256, 8, 8), (512, 4, 16), (256, 2, 64)])
def test_zigzag_work_is_balanced_in_closed_form(L, P, block):
    c = L // (2 * P)
    Tc = c // block
    z = oracle.shard_work(L, P, block, "zigzag", causal=True)
    for i in range(P):
        assert z["pairs"][i] == c * c * (2 * P - 1) + c * (c + 1)
        assert z["tiles"][i] == Tc * Tc * (2 * P - 1) + Tc * (Tc + 1)
    assert sum(z["pairs"]) == L * (L + 1) // 2
    assert len(set(z["visits"])) == 1


def test_striped_balance_at_the_workload_shapes():
    # max/mean of unmasked pairs per shard, striped, from the closed form above
    for L, P in ((8192, 8), (32768, 8), (262144, 16), (1048576, 32)):
        n = L // P
        pairs = [P * n * (n - 1) // 2 + n * (i + 1) for i in range(P)]
        assert max(pairs) / (sum(pairs) / P) <= 1.05


def test_tile_class_follows_block_rule():
    # contiguous blocks of 4 tokens: later KV block -> skip, same -> diag, earlier -> full
    q_blk = list(range(8, 12))
    assert oracle.tile_class(q_blk, list(range(12, 16)), True) == "skip"
    assert oracle.tile_class(q_blk, list(range(8, 12)), True) == "diag"
    assert oracle.tile_class(q_blk, list(range(4, 8)), True) == "full"
    assert oracle.tile_class(q_blk, list(range(12, 16)), False) == "full"
