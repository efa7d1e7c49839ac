"""Shard assignment, ring order and the per-shard causal work model (pure Python).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Assignment of token t (0-based, natural order) to one of P shards of n = L/P tokens:
* contiguous -- shard t div n, local index t mod n (vanos001, section "Ring Attention:
  Compute While You Communicate": device i owns the i-th slice of the sequence);
* striped    -- shard t mod P, local index t div P (vanos001, section "The Causal-Mask
  Problem: Striped Attention": row r goes to device r mod P);
* zigzag     -- the sequence is cut into 2P chunks of c = L/(2P) tokens and shard i holds
  chunks i and 2P-1-i, in that order (vanos001, same section: each device gets two
  half-blocks placed symmetrically near the start and the end of the sequence).  Local
  index a < c is token i*c + a, local index a >= c is token (2P-1-i)*c + (a - c).

Ring order (labhub, section "リング通信パターン"; vanos001 ring diagram): at step k
shard i works on the KV shard (i - k) mod P, so shard 0 sees 0, P-1, P-2, ..., 1.

Work units for shard i (the vanos001 "Worked Demo" counts unmasked KV-block visits):
  tiles    -- (Q block, KV block) pairs of `block` x `block` tokens, taken over the
              ring schedule, in which at least one (query, key) pair is unmasked;
  pairs    -- unmasked (query, key) pairs whose query lives on shard i;
  visits   -- the demo's own unit: for every query row of shard i, the number of
              natural-order KV blocks of `block` keys holding at least one unmasked
              key (row div block + 1 when causal, L / block otherwise).
All three are computed here by enumeration from the definitions; the tests check them
against closed forms and against the printed demo output.
"""

CONTIGUOUS = "contiguous"
STRIPED = "striped"
ZIGZAG = "zigzag"


def _check_layout(layout):
    if layout not in (CONTIGUOUS, STRIPED, ZIGZAG):
        raise ValueError("layout must be 'contiguous', 'striped' or 'zigzag'")


def shard_of(t, L, P, layout):
    _check_layout(layout)
    n = L // P
    if layout == ZIGZAG:
        ch = t // (L // (2 * P))
        return ch if ch < P else 2 * P - 1 - ch
    return t // n if layout == CONTIGUOUS else t % P


def local_of(t, L, P, layout):
    _check_layout(layout)
    n = L // P
    if layout == ZIGZAG:
        c = L // (2 * P)
        return t % c if t // c < P else c + t % c
    return t % n if layout == CONTIGUOUS else t // P


def shard_tokens(i, L, P, layout):
    """Natural-order token indices held by shard i, in local order."""
    _check_layout(layout)
    n = L // P
    if layout == CONTIGUOUS:
        return list(range(i * n, (i + 1) * n))
    if layout == ZIGZAG:
        c = L // (2 * P)
        return list(range(i * c, (i + 1) * c)) + list(range((2 * P - 1 - i) * c, (2 * P - i) * c))
    return [a * P + i for a in range(n)]


def ring_order(i, P):
    """KV shards visited by shard i over steps k = 0..P-1: (i - k) mod P."""
    return [(i - k) % P for k in range(P)]


def tile_class(q_tokens, k_tokens, causal):
    """'skip' / 'full' / 'diag' for one Q block against one KV block.

    Decided from original token positions: 'skip' when every pair is masked, 'full'
    when none is, 'diag' otherwise (labhub section "Causal Masking の処理": a KV block
    after the query block is skipped, the same block is masked, earlier ones are not).
    """
    if not causal:
        return "full"
    vis = [[kt <= qt for kt in k_tokens] for qt in q_tokens]
    n_vis = sum(sum(row) for row in vis)
    if n_vis == 0:
        return "skip"
    if n_vis == len(q_tokens) * len(k_tokens):
        return "full"
    return "diag"


def shard_work(L, P, block, layout, causal):
    """Per-shard work in the three units above. Returns dict of lists of ints."""
    _check_layout(layout)
    if L % P or (L // P) % block:
        raise ValueError("seq_len must be divisible by P * block")
    if layout == ZIGZAG and (L % (2 * P) or (L // (2 * P)) % block):
        raise ValueError("zigzag needs seq_len divisible by 2 * P * block")
    n = L // P
    T = n // block
    tokens = [shard_tokens(i, L, P, layout) for i in range(P)]
    # earliest and latest token of every block (a block pair is computed iff its
    # earliest key is not after its latest query, i.e. some pair is unmasked)
    first = [[min(tokens[i][u * block:(u + 1) * block]) for u in range(T)]
             for i in range(P)]
    last = [[max(tokens[i][u * block:(u + 1) * block]) for u in range(T)]
            for i in range(P)]
    tiles = [0] * P
    pairs = [0] * P
    visits = [0] * P
    for i in range(P):
        for t in range(T):
            for j in ring_order(i, P):
                for u in range(T):
                    if not causal or first[j][u] <= last[i][t]:
                        tiles[i] += 1
        for r in tokens[i]:
            pairs[i] += (r + 1) if causal else L
            visits[i] += (r // block + 1) if causal else (L // block)
    return {"tiles": tiles, "pairs": pairs, "visits": visits}
