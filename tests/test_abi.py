"""Host-only tests of the C ABI: the library loads, exports every declared symbol, rejects
bad arguments before any launch, and its closed-form work model matches the oracle's
enumeration and the printed demo.  No GPU is needed (no compute call reaches CUDA)."""

import ctypes
import os

import pytest

import oracle
import exact_blockwise_ring_gb300 as era
from exact_blockwise_ring_gb300 import api

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(api.LIB_PATH):
        from exact_blockwise_ring_gb300 import build
        build.build()
    return api.lib()


def test_exports_every_declared_symbol(L):
    names = api.header_symbols()
    assert "ra_fwd" in names and "ra_bwd" in names and "ra_merge" in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code, name in api.STATUS.items():
        assert L.ra_status_string(code).decode() == name


def _params(**kw):
    base = dict(batch=1, seq_len=1024, heads=2, head_dim=128, P=4, block=128, layout=0,
                causal=1, softmax_scale=0.0, n_split=0, kv_heads=0)
    base.update(kw)
    return api.Params(base["batch"], base["seq_len"], base["heads"], base["head_dim"],
                      base["block"], base["P"], base["layout"], base["causal"],
                      base["softmax_scale"], base["n_split"], base["kv_heads"])


FAKE = ctypes.c_void_p(1 << 20)      # 16-byte aligned, never dereferenced on these paths


def _fwd(L, prm, q=FAKE, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 30, odt=0, sw=None):
    return L.ra_fwd(ctypes.byref(prm), q, FAKE, FAKE, out, odt, lse, sw, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(seq_len=1000), 1),              # not divisible by P * block
    (dict(batch=0), 1),
    (dict(seq_len=0), 1),                 # empty sequence
    (dict(seq_len=-1024), 1),
    (dict(seq_len=1 << 33, heads=1024, P=8), 1),   # past the 2^40-element guard
    (dict(heads=0), 1),
    (dict(P=0), 1),
    (dict(P=2000, seq_len=2000 * 128), 1),
    (dict(head_dim=96), 2),               # valid, no kernel
    (dict(block=64, seq_len=1024), 2),
    (dict(layout=3), 1),
    (dict(layout=2, seq_len=4 * 128 * 3), 1),   # zigzag: L / P not a multiple of 2 * block
    (dict(causal=3), 1),
    (dict(softmax_scale=-1.0), 1),
    (dict(softmax_scale=float("inf")), 1),
    (dict(n_split=3), 1),                 # not a divisor of P
    (dict(heads=6, kv_heads=4), 1),       # kv_heads must divide heads
    (dict(kv_heads=-1), 1),
])
def test_fwd_rejects_bad_params(L, kw, code):
    assert _fwd(L, _params(**kw)) == code
    assert L.ra_last_error_message().decode()


def test_fwd_rejects_bad_pointers_and_workspace(L):
    prm = _params()
    assert _fwd(L, prm, q=None) == 1
    assert _fwd(L, prm, out=ctypes.c_void_p((1 << 20) + 8)) == 1
    assert _fwd(L, prm, odt=7) == 1
    assert _fwd(L, prm, ws=None) == 3
    assert _fwd(L, prm, ws_bytes=16) == 3
    assert _fwd(L, prm, sw=ctypes.c_void_p((1 << 20) + 4)) == 1


def test_bwd_rejects_bad_arguments(L):
    prm = _params()
    args = [FAKE] * 3 + [FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None]
    assert L.ra_bwd(ctypes.byref(_params(seq_len=1000)), *args) == 1
    assert L.ra_bwd(ctypes.byref(_params(head_dim=96)), *args) == 2     # valid, no kernel
    bad = list(args)
    bad[7] = None                                            # dq
    assert L.ra_bwd(ctypes.byref(prm), *bad) == 1
    bad = list(args)
    bad[11] = 64                                             # workspace too small
    assert L.ra_bwd(ctypes.byref(prm), *bad) == 3


def test_merge_rejects_bad_arguments(L):
    assert L.ra_merge(0, FAKE, FAKE, 1, 128, 1, 128, FAKE, 0, FAKE, None) == 1
    assert L.ra_merge(2, FAKE, FAKE, 1, 128, 1, 12, FAKE, 0, FAKE, None) == 1
    assert L.ra_merge(2, None, FAKE, 1, 128, 1, 128, FAKE, 0, FAKE, None) == 1


def test_workspace_sizes(L):
    prm = _params(seq_len=32768, heads=32, P=8, n_split=1)
    assert api.fwd_workspace_bytes(prm) == 256
    b = api.bwd_workspace_bytes(prm)
    assert b >= 256 + 32768 * 32 * 128 * 4 + 32 * 32768 * 4
    assert api.fwd_workspace_bytes(_params(seq_len=1000)) == 0
    split = api.fwd_workspace_bytes(_params(seq_len=512, heads=2, head_dim=64, n_split=4))
    assert split >= 256 + 4 * (512 * 2 * 64 * 4 + 2 * 512 * 4)


def test_selftest_rejects_bad_arguments(L):
    assert L.ra_selftest_timeout(None, 256, 100, None) == 3
    assert L.ra_selftest_timeout(FAKE, 256, 0, None) == 1


# ---- host work model against the oracle --------------------------------------------

def test_work_model_reproduces_demo(L):
    rows = {}
    for ln in open(os.path.join(GOLDEN, "work_demo.txt")):
        if ln.strip() and not ln.startswith("#"):
            f = ln.split()
            rows[f[0]] = [int(x) for x in f[1:5]]
    for layout in ("contiguous", "striped"):
        w = era.ra_shard_work_model(32, 4, 8, layout, True)
        assert w["visits"] == rows[layout]


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("L_,P,block", [(64, 4, 4), (512, 8, 16), (1024, 2, 128), (2048, 4, 256),
                                        (96, 3, 4)])
def test_work_model_matches_oracle(L, layout, causal, L_, P, block):
    got = era.ra_shard_work_model(L_, P, block, layout, causal)
    want = oracle.shard_work(L_, P, block, layout, causal)
    assert got == want


def test_work_model_matches_oracle_random_shapes(L):
    # seeded sweep of small shapes: any P, any number of blocks per shard (zigzag: an even
    # number), blocks of 1 to 16 tokens, every layout, causal or not
    import random
    rng = random.Random(20261202)
    for _ in range(200):
        layout = rng.choice(["contiguous", "striped", "zigzag"])
        causal = rng.random() < 0.8
        P = rng.randint(1, 9)
        block = rng.choice([1, 2, 3, 4, 8, 16])
        T = rng.randint(1, 6) * (2 if layout == "zigzag" else 1)
        L_ = P * T * block
        got = era.ra_shard_work_model(L_, P, block, layout, causal)
        want = oracle.shard_work(L_, P, block, layout, causal)
        assert got == want, (L_, P, block, layout, causal)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "LIB_PATH", str(tmp_path / "libra.so"))
    with pytest.raises(RuntimeError, match="not built"):
        api.lib()


# ---- blockwise transformer layer: host-side argument checks ------------------------

def test_linear_rejects_bad_arguments(L):
    ok = (256, 128, 256, FAKE, FAKE, FAKE, None, 0, FAKE, FAKE, 256, None)
    bad = list(ok)
    bad[0] = 200                                            # rows % 128
    assert L.ra_linear(*bad) == 2
    bad = list(ok)
    bad[2] = 300                                            # out_features % 256
    assert L.ra_linear(*bad) == 2
    bad = list(ok)
    bad[7] = 2                                              # residual epilogue, no residual
    assert L.ra_linear(*bad) == 1
    bad = list(ok)
    bad[7] = 9
    assert L.ra_linear(*bad) == 1
    bad = list(ok)
    bad[10] = 16                                            # workspace too small
    assert L.ra_linear(*bad) == 3
    bad = list(ok)
    bad[3] = ctypes.c_void_p((1 << 20) + 8)                 # misaligned x
    assert L.ra_linear(*bad) == 1


def test_layernorm_rejects_bad_arguments(L):
    assert L.ra_layernorm(4, 500, FAKE, FAKE, FAKE, 1e-5, FAKE, 0, None) == 2
    assert L.ra_layernorm(4, 512, FAKE, FAKE, FAKE, 0.0, FAKE, 0, None) == 1
    assert L.ra_layernorm(4, 512, FAKE, FAKE, FAKE, 1e-5, FAKE, 5, None) == 1
    assert L.ra_layernorm(4, 512, None, FAKE, FAKE, 1e-5, FAKE, 0, None) == 1


@pytest.mark.parametrize("kw,ok", [
    (dict(), True),
    (dict(heads=2), False),                 # d_model 256: not a multiple of 512
    (dict(d_ff=1000), False),
    (dict(block_rows=100), False),
    (dict(kv_heads=2), True),               # grouped-query: K, V 256 wide
    (dict(kv_heads=1), False),              # K, V 128 wide: not a multiple of 256
    (dict(kv_heads=3), False),              # not a divisor of heads
    (dict(seq_len=1000), False),            # invalid attention parameters
])
def test_bpt_workspace_bytes_validates(L, kw, ok):
    base = dict(batch=1, seq_len=1024, heads=4, head_dim=128, d_ff=1024, P=4, block=128,
                block_rows=256, kv_heads=0)
    base.update(kw)
    prm = era.make_bpt_params(base["batch"], base["seq_len"], base["heads"], base["head_dim"],
                              base["d_ff"], base["P"], base["block"], "striped", True,
                              base["block_rows"])
    prm.attn.kv_heads = base["kv_heads"]
    n = era.bpt_workspace_bytes(prm)
    if ok:
        d = base["heads"] * base["head_dim"]
        rows = base["batch"] * base["seq_len"]
        dkv = (base["kv_heads"] or base["heads"]) * base["head_dim"]
        assert n >= (2 * d + 2 * dkv) * rows * 2 + base["block_rows"] * (d * 6 + base["d_ff"] * 2)
    else:
        assert n == 0


def test_layer_bindings_check_their_inputs_before_any_call():
    import torch
    x = torch.zeros((128, 64), dtype=torch.bfloat16)          # a CPU tensor: refused
    w = torch.zeros((256, 64), dtype=torch.bfloat16)
    b = torch.zeros(256)
    with pytest.raises(ValueError, match="CUDA"):
        era.ra_linear(x, w, b)
    with pytest.raises(ValueError, match="CUDA"):
        era.ra_layernorm(torch.zeros((4, 512)), torch.ones(512), torch.zeros(512))
    with pytest.raises(ValueError, match="CUDA"):
        era.ra_bpt_fwd(torch.zeros((1, 1024, 512), dtype=torch.bfloat16), {}, 4, 4, 128)


def test_bpt_train_workspace_and_backward_checks(L):
    prm = era.make_bpt_params(1, 1024, 4, 128, 1024, 4, 128, "striped", True, 256)
    assert era.bpt_train_workspace_bytes(prm) > era.bpt_workspace_bytes(prm) > 0
    # head_dim 64 has a backward too; d_model 8192 > 4096 has a forward but no backward
    p64 = era.make_bpt_params(1, 1024, 8, 64, 1024, 4, 128, "striped", True, 256)
    assert era.bpt_train_workspace_bytes(p64) > era.bpt_workspace_bytes(p64) > 0
    big = era.make_bpt_params(1, 1024, 64, 128, 1024, 4, 128, "striped", True, 256)
    assert era.bpt_workspace_bytes(big) > 0 and era.bpt_train_workspace_bytes(big) == 0
    w = api.BptWeights(*([FAKE.value] * len(api.BPT_WEIGHTS)))
    gr = api.BptGrads(*([FAKE.value] * (1 + len(api.BPT_WEIGHTS))))
    assert L.ra_bpt_bwd(ctypes.byref(big), FAKE, ctypes.byref(w), FAKE, ctypes.byref(gr), FAKE,
                        1 << 40, None) == 2
    gr_null = api.BptGrads(*([None] + [FAKE.value] * len(api.BPT_WEIGHTS)))
    assert L.ra_bpt_bwd(ctypes.byref(prm), FAKE, ctypes.byref(w), FAKE, ctypes.byref(gr_null),
                        FAKE, 1 << 40, None) == 1
    assert L.ra_bpt_bwd(ctypes.byref(prm), FAKE, ctypes.byref(w), FAKE, ctypes.byref(gr), FAKE,
                        64, None) == 3


def _documented_valid(B, L, H, D, blk, P, layout, causal, scale, n_split, kv):
    """The rules ra.h states for ra_params_t, restated."""
    if B < 1 or H < 1 or L < 1 or not 1 <= P <= 1024:
        return False
    if layout not in (0, 1, 2) or causal not in (0, 1):
        return False
    if D not in (64, 128) or blk not in (128, 256):
        return False
    if L % (P * blk) or (layout == 2 and L % (2 * P * blk)):
        return False
    if not (scale >= 0.0) or scale == float("inf"):
        return False
    if n_split < 0 or (n_split > 0 and P % n_split):
        return False
    if kv < 0 or (kv > 0 and H % kv):
        return False
    return B * L * H * D <= 1 << 40 and B * H * L <= 1 << 36


def test_parameter_rules_match_the_header(L):
    # seeded sweep over valid and invalid parameter sets: the library accepts exactly the
    # ones the header's rules allow (workspace size 0 marks a rejected set)
    import random
    rng = random.Random(4242)
    seen = {True: 0, False: 0}
    def pick(good, bad, p_good=0.9):
        return rng.choice(good) if rng.random() < p_good else rng.choice(bad)

    for _ in range(3000):
        P = pick([1, 2, 3, 4, 8, 16, 1024], [0, -1, 1025])
        blk = pick([128, 256], [64, 100, 0])
        layout = pick([0, 1, 2], [3, -1])
        mult = rng.choice([1, 2, 3, 4, 6])
        L_ = max(P, 1) * max(blk, 1) * mult
        if rng.random() < 0.15:
            L_ += rng.choice([1, 64, 128])
        if rng.random() < 0.03:
            L_ = rng.choice([0, -128, 1 << 34])
        B = pick([1, 2, 3], [0, -1, 1 << 20])
        H = pick([1, 2, 6, 32], [0, -4])
        D = pick([64, 128], [96, 0, 256])
        causal = pick([0, 1], [2, -1])
        scale = pick([0.0, 0.125, 3.0], [-1.0, float("inf"), float("nan")])
        n_split = pick([0, 1, 2, 4], [3, -1, 5])
        kv = pick([0, 1, 2], [3, -2, 4, 5])
        prm = api.Params(B, L_, H, D, blk, P, layout, causal, scale, n_split, kv)
        want = _documented_valid(B, L_, H, D, blk, P, layout, causal, scale, n_split, kv)
        got = api.fwd_workspace_bytes(prm) > 0
        assert got == want, (B, L_, H, D, blk, P, layout, causal, scale, n_split, kv)
        seen[want] += 1
    assert seen[True] > 100 and seen[False] > 100


def test_layer_parameter_rules_match_the_header(L):
    # the layer's own rules on top of the attention's (a valid attention part throughout):
    # d_model % 512 == 0 and <= 8192, H_kv * head_dim % 256 == 0, d_ff a positive multiple
    # of 256, block_rows 0 or a positive multiple of 128, ln_eps >= 0; the training
    # workspace also needs d_model <= 4096
    import random
    rng = random.Random(515)
    seen = {True: 0, False: 0}
    for _ in range(1500):
        D = rng.choice([64, 128])
        H = rng.choice([1, 2, 4, 6, 8, 16, 32, 48, 64, 65, 96, 128])
        kv = rng.choice([0, 0, 1, 2, 4, 8])
        if kv and H % kv:
            kv = 0
        d_ff = rng.choice([256, 512, 4096, 16384, 0, 100, 300])
        block_rows = rng.choice([0, 128, 256, 16384, 100, -128])
        eps = rng.choice([0.0, 1e-5, 1e-6, -1.0, float("nan")])
        attn = api.Params(1, 1024, H, D, 128, 4, 1, 1, 0.0, 0, kv)
        prm = api.BptParams(attn, d_ff, block_rows, eps)
        d, dkv = H * D, (kv or H) * D
        want = (d % 512 == 0 and d <= 8192 and dkv % 256 == 0 and d_ff >= 256 and
                d_ff % 256 == 0 and block_rows >= 0 and block_rows % 128 == 0 and eps >= 0.0)
        assert (api.lib().ra_bpt_workspace_bytes(ctypes.byref(prm)) > 0) == want, (
            H, D, kv, d_ff, block_rows, eps)
        want_train = want and d <= 4096
        assert (api.lib().ra_bpt_train_workspace_bytes(ctypes.byref(prm)) > 0) == want_train
        seen[want] += 1
    assert seen[True] > 50 and seen[False] > 50


def test_checked_build_links_and_exports_the_same_symbols(tmp_path):
    """The checked build (compiled with RA_CHECKS) links, reports itself as checked and
    exports every symbol the header declares; the normal build reports no checks."""
    import ctypes
    import shutil
    from exact_blockwise_ring_gb300 import build
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("needs nvcc")
    path = build.build(checked=True)
    h = ctypes.CDLL(path)
    h.ra_checks_enabled.restype = ctypes.c_int
    assert h.ra_checks_enabled() == 1
    for name in api.header_symbols():
        assert hasattr(h, name), name
    if not os.environ.get("RA_LIBRARY"):
        assert api.lib().ra_checks_enabled() == 0
