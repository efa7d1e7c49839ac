"""CPU fp64 oracle for exact blockwise ring attention (contiguous, striped and zigzag).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything in this package.  The
product path (the CUDA library and its Python binding) never imports it, and this
package imports nothing from the product path.

Sources (four web pages on Ring Attention and Striped Attention):

* "Ring Attention 論文分析" (labhub): the BPT blockwise online softmax
  (section "ブロック単位の分割戦略"), the ring forward (section "リングトポロジーと
  KV の循環"), causal block skipping (section "Causal Masking の処理"), the ring
  order (section "リング通信パターン") and the backward formulas (section
  "逆伝播での KV 再循環").
* "Ring Attention: Sequence Parallelism for Long Context" (vanos001): the ring
  diagram, the striped assignment (section "The Causal-Mask Problem: Striped
  Attention") and the worked demo of per-device work (section "Worked Demo").
* the same labhub page, section "BPT の Feedforward 融合": the blockwise transformer
  layer (attention fused with the feed-forward network per query block).
* "Sequence parallelism and ring attention" (aiunderstanding) and the Striped
  Attention summary (aibr.jp, section 3, permutation equivariance).

Modules:
    attention -- exact attention forward/backward by its definition (row-blocked
                 full-row softmax, no online merge, no ring) and a brute-force
                 pure-Python version for tiny inputs.
    ring      -- an fp64 emulator of the ring schedule with online softmax and the
                 partial merge, used only to test invariants ("ring == full").
    work      -- shard assignment, ring order and the per-shard work model.
    gqa       -- grouped-query attention (fewer key/value heads than query heads) on top
                 of ``attention``.
    bpt       -- one Blockwise Parallel Transformer layer (projections, attention, output
                 projection, residuals, LayerNorms, GELU feed-forward), forward and
                 backward.

Parity status: every function here is pinned by tests in ``tests/test_oracle_*.py``
against things other than itself (a library softmax attention, closed forms,
finite differences, the pages' printed demo output).  None is "parity unpinned".
"""

from .attention import (attention_fwd, attention_bwd, attention_rows_fwd, attention_rows_dq,
                        attention_cols_dkdv, brute_force_fwd, default_scale)
from .ring import ring_fwd, ring_partials, merge_partials
from .work import (shard_of, local_of, shard_tokens, ring_order, shard_work,
                   tile_class)
from .gqa import gqa_fwd, gqa_bwd, gqa_cols_dkdv, group_size
from .bpt import (bpt_layer_bwd, bpt_layer_fwd, bpt_layer_fwd_blocked, bpt_layer_rows, gelu,
                  gelu_grad, layer_norm, layer_norm_bwd)

__all__ = [
    "attention_fwd", "attention_bwd", "attention_rows_fwd", "attention_rows_dq",
    "attention_cols_dkdv", "brute_force_fwd",
    "default_scale", "ring_fwd", "ring_partials", "merge_partials", "shard_of",
    "local_of", "shard_tokens", "ring_order", "shard_work", "tile_class", "gqa_fwd", "gqa_bwd", "gqa_cols_dkdv",
    "group_size", "bpt_layer_fwd", "bpt_layer_fwd_blocked", "bpt_layer_rows", "bpt_layer_bwd",
    "gelu", "gelu_grad", "layer_norm", "layer_norm_bwd",
]
