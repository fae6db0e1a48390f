"""CPU oracle (test infrastructure only; see ``oracle.csa2``)."""
from .csa2 import (FULL, REINDEX, REUSE, SWA, to_f64, round_bf16, indexer_scores, block_keys,
                   select_topk, pool_blocks, pooled_entries, layer_indices, attend,
                   sparse_attention, run_group, group_counts, kv_append, swa_append)

__all__ = ["FULL", "REINDEX", "REUSE", "SWA", "to_f64", "round_bf16", "indexer_scores", "block_keys",
           "select_topk", "pool_blocks", "pooled_entries", "layer_indices", "attend",
           "sparse_attention", "run_group", "group_counts", "kv_append", "swa_append"]
