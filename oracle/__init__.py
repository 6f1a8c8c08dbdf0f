"""fp64 CPU oracles for the fused attention forward (with and without
dropout), the projection GEMM around it and the layer slice they form (test
infrastructure only).

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  The library never does.
"""
from .attention_fp64 import (attention, attention_head, attention_rows, attention_split,
                        combine_partials, kv_head_of)
from .dropout_fp64 import attention_dropout, attention_dropout_rows, drop_threshold, keep_mask
from .gemm_fp64 import gemm_nt, gemm_nt_rows
from .layer_fp64 import layer, layer_rows, merge_heads, round_bf16, split_heads

__all__ = ["attention", "attention_head", "attention_rows", "attention_split",
           "combine_partials", "kv_head_of", "gemm_nt", "gemm_nt_rows",
           "layer", "layer_rows", "merge_heads", "round_bf16", "split_heads",
           "attention_dropout", "attention_dropout_rows", "drop_threshold", "keep_mask"]
