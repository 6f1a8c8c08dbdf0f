"""fp64 CPU oracle for the fused attention forward (test infrastructure only).

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  The library never does.
"""
from .attention_fp64 import (attention, attention_head, attention_rows, attention_split,
                        combine_partials, kv_head_of)

__all__ = ["attention", "attention_head", "attention_rows", "attention_split",
           "combine_partials", "kv_head_of"]
