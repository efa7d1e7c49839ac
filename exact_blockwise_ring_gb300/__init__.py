"""Exact blockwise ring attention (contiguous, striped and zigzag layouts; multi-head or
grouped-query) for NVIDIA GB300 (sm_103a).

The computation lives in libra.so (C ABI: include/ra.h), built from csrc/ by
``exact_blockwise_ring_gb300.build.build()``; this package only marshals arguments.
"""

from .api import (BPT_WEIGHTS, LAYOUTS, BptGrads, BptLayer, BptParams, BptWeights, Params,
                  RaError, RingAttention, Workspace, bpt_train_workspace_bytes,
                  bpt_workspace_bytes, bwd_workspace_bytes, fwd_workspace_bytes,
                  header_symbols, lib, make_bpt_params, make_params, ra_bpt_bwd, ra_bpt_fwd, ra_bwd,
                  ra_bwd_stages, ra_fwd, ra_layernorm, ra_linear, ra_merge, ra_selftest_exp2,
                  ra_selftest_timeout,
                  ra_shard_work_model, ring_attention)

__all__ = ["BPT_WEIGHTS", "LAYOUTS", "BptGrads", "BptLayer", "BptParams", "BptWeights", "Params",
           "RaError", "RingAttention", "Workspace", "bpt_train_workspace_bytes",
           "bpt_workspace_bytes", "bwd_workspace_bytes", "fwd_workspace_bytes", "header_symbols",
           "lib", "make_bpt_params", "make_params", "ra_bpt_bwd", "ra_bpt_fwd", "ra_bwd", "ra_bwd_stages", "ra_fwd", "ra_layernorm", "ra_linear",
           "ra_merge", "ra_selftest_exp2", "ra_selftest_timeout", "ra_shard_work_model", "ring_attention"]
