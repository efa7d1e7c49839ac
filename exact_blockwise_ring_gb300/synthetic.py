"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

Recipe: Q, K, V and the upstream gradient dO are drawn, in that order, as N(0, 1)
float32 from one ``torch.Generator`` seeded with ``seed``, shape [B, L, H, D], and
rounded to bfloat16 (round to nearest even).  The oracle receives the same rounded
values widened to float64.  This module holds no attention arithmetic.
"""

import torch

# The workloads of this library's test and benchmark plan.
WORKLOADS = {
    "tiny":  dict(batch=1, heads=2, head_dim=64, seq_len=512, P=4, block=128,
                  causal=False, layouts=("contiguous",), backward=False),
    "8k":    dict(batch=1, heads=8, head_dim=128, seq_len=8192, P=8, block=128,
                  causal=True, layouts=("contiguous", "striped", "zigzag"), backward=False),
    "32k":   dict(batch=1, heads=32, head_dim=128, seq_len=32768, P=8, block=128,
                  causal=True, layouts=("striped", "zigzag"), backward=True),
    "262k":  dict(batch=1, heads=32, head_dim=128, seq_len=262144, P=16, block=256,
                  causal=True, layouts=("striped", "zigzag"), backward=True),
    "1m":    dict(batch=1, heads=8, head_dim=128, seq_len=1048576, P=32, block=256,
                  causal=True, layouts=("striped", "contiguous", "zigzag"), backward=True),
    # grouped-query attention: 32 query heads on 8 key/value heads (4 per group)
    "32k-gqa": dict(batch=1, heads=32, kv_heads=8, head_dim=128, seq_len=32768, P=8,
                    block=128, causal=True, layouts=("zigzag", "striped"), backward=True),
    # head dim 64 at the 32k workload's width: 64 heads of 64
    "32k-d64": dict(batch=1, heads=64, head_dim=64, seq_len=32768, P=8, block=128,
                    causal=True, layouts=("zigzag", "striped"), backward=True),
    # one blockwise transformer layer (forward): d_model 4096 = 32 x 128, d_ff = 4 d_model,
    # the feed-forward part in blocks of 16384 rows
    "32k-bpt": dict(batch=1, heads=32, head_dim=128, seq_len=32768, P=8, block=128,
                    causal=True, layouts=("zigzag", "striped"), backward=False, d_ff=16384,
                    block_rows=16384),
}

SEEDS = {"tiny": 1000, "8k": 1001, "32k": 1002, "262k": 1003, "1m": 1004, "32k-gqa": 1005,
         "32k-bpt": 1006, "32k-d64": 1007}


def make_inputs(batch, seq_len, heads, head_dim, seed, device="cpu", with_dout=True,
                kv_heads=None):
    """Return (q, k, v[, dout]) bfloat16 tensors on ``device``: q and dout
    [B, L, heads, D], k and v [B, L, kv_heads, D] (kv_heads defaults to heads).

    The generator lives on ``device``; CPU and CUDA streams of numbers differ, so
    a test that compares against the oracle generates on the CPU (or copies device
    tensors to the host) and hands the same tensors to both sides.
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    hq = heads
    hkv = heads if kv_heads is None else kv_heads
    names = ("q", "k", "v", "dout") if with_dout else ("q", "k", "v")
    out = []
    for nm in names:
        h = hkv if nm in ("k", "v") else hq
        x = torch.randn((batch, seq_len, h, head_dim), generator=g, device=device,
                        dtype=torch.float32)
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def make_bpt_weights(d, d_ff, seed, device="cpu", d_kv=None):
    """Random parameters of one blockwise transformer layer: Linear weights [out, in] drawn
    N(0, 1/in) and rounded to bf16, biases N(0, 0.01) fp32, LayerNorm scales 1 + N(0, 0.01)
    and shifts N(0, 0.01) fp32 (N(mean, variance)), drawn in the order wq, wk, wv, wo, w1, w2,
    bq, bk, bv, bo, b1, b2, ln1 scale, ln1 shift, ln2 scale, ln2 shift."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    d_kv = d if d_kv is None else d_kv        # K, V projection width (grouped-query: < d)
    shapes = {"wq": (d, d), "wk": (d_kv, d), "wv": (d_kv, d), "wo": (d, d), "w1": (d_ff, d),
              "w2": (d, d_ff)}
    w = {}
    for name, (o, i) in shapes.items():
        x = torch.randn((o, i), generator=g, device=device, dtype=torch.float32) / (i ** 0.5)
        w[name] = x.to(torch.bfloat16)
    for name, n in (("bq", d), ("bk", d_kv), ("bv", d_kv), ("bo", d), ("b1", d_ff), ("b2", d)):
        w[name] = 0.1 * torch.randn(n, generator=g, device=device, dtype=torch.float32)
    for ln in ("ln1", "ln2"):
        w[ln + "_g"] = 1.0 + 0.1 * torch.randn(d, generator=g, device=device, dtype=torch.float32)
        w[ln + "_b"] = 0.1 * torch.randn(d, generator=g, device=device, dtype=torch.float32)
    return w


def to_f64(*tensors):
    """bfloat16 torch tensors -> float64 NumPy arrays (exact widening)."""
    return tuple(t.detach().to("cpu", torch.float64).numpy() for t in tensors)
