"""fp64 CPU oracle for the projection GEMM around attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
the tests and the CPU-baseline leg of ``bench.py`` call it.  It shares no
code with the CUDA path.

What it computes is the plain definition of the projections that feed and
drain the attention forward (the QKV and O projections of the decoder chain
on "CS149 L11: Programming Specialized Hardware", section 6, and the matrix
multiply kernel of its section 4): for inputs X [M, K] and a weight W [N, K]
stored row-major as a linear layer keeps it,

    C[m, n] = sum_k X[m, k] * W[n, k]          (C = X W^T)

on the bf16-exact input values upcast to fp64.  A library matrix product is
the one step (the blocking, tiling and accumulation order of the GPU kernel
are its own business and change only rounding).
"""
from __future__ import annotations

import numpy as np


def gemm_nt(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """C = A B^T in fp64; a [M, K], b [N, K] (any float dtype, upcast exactly)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("gemm_nt wants a [M, K] and b [N, K], got %s and %s" % (a.shape, b.shape))
    return a @ b.T


def gemm_nt_rows(a: np.ndarray, b: np.ndarray, rows) -> np.ndarray:
    """Rows `rows` of A B^T only (for sampled checks of large products)."""
    return gemm_nt(np.asarray(a)[list(rows)], b)
