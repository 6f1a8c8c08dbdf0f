"""fp64 CPU oracles for the fused attention forward and the projection GEMM
around it (test infrastructure only).

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  The library never does.
"""
from .attention_fp64 import (attention, attention_head, attention_rows, attention_split,
                        combine_partials, kv_head_of)
from .gemm_fp64 import gemm_nt, gemm_nt_rows

__all__ = ["attention", "attention_head", "attention_rows", "attention_split",
           "combine_partials", "kv_head_of", "gemm_nt", "gemm_nt_rows"]
