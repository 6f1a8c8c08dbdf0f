"""fp64 CPU oracle for one attention layer slice: QKV projection, attention,
output projection.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
the tests and the CPU-baseline leg of ``bench.py`` call it.  It shares no
code with the CUDA path.

What it computes is the part of the decoder-layer chain on "CS149 L11:
Programming Specialized Hardware" (section 6: Q/K/V GEMMs, Q K^T, scale,
mask, softmax, x V, the O GEMM) that surrounds the fused attention, as three
plain steps on the bf16-exact inputs upcast to fp64:

    QKV = X W_qkv^T                      (gemm_fp64.gemm_nt)
    Q, K, V = the column blocks of QKV   (Hq heads of Q, then Hkv of K, then
                                          Hkv of V, d features each)
    O = attention(Q, K, V)               (attention_fp64.attention)
    Y = O W_o^T                          (O with its heads side by side again)

Reading where the pages are silent: a layer hands its intermediates from one
kernel to the next in the kernels' input type, bf16.  So QKV and O are
rounded to bf16 (to nearest, ties to even) before they are used, as the GPU
path stores them; ``round_intermediates=False`` gives the exact fp64 chain.

Pinned by tests/test_oracle_layer.py (reductions to plain attention under
identity-like weights, grouped-query slicing, a pure-Python brute force,
exact linearity, and the bf16 rounding against exact ties and a library
conversion).
"""
from __future__ import annotations

import numpy as np

from .attention_fp64 import attention, attention_head, kv_head_of
from .gemm_fp64 import gemm_nt


def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (8 significant bits), ties
    to even, returned as fp64.  Values stay in bf16's normal range here."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def split_heads(qkv, B: int, N: int, Hq: int, Hkv: int, d: int):
    """Q [B, Hq, N, d], K and V [B, Hkv, N, d] from QKV rows [B*N, (Hq+2Hkv)*d]."""
    qkv = np.asarray(qkv).reshape(B, N, Hq + 2 * Hkv, d)
    q = qkv[:, :, :Hq].transpose(0, 2, 1, 3)
    k = qkv[:, :, Hq:Hq + Hkv].transpose(0, 2, 1, 3)
    v = qkv[:, :, Hq + Hkv:].transpose(0, 2, 1, 3)
    return q, k, v


def merge_heads(o) -> np.ndarray:
    """O [B, Hq, N, d] back to token rows [B*N, Hq*d]."""
    B, Hq, N, d = o.shape
    return np.asarray(o).transpose(0, 2, 1, 3).reshape(B * N, Hq * d)


def layer(x, w_qkv, w_o, B: int, N: int, Hq: int, Hkv: int, causal: bool, scale: float,
          round_intermediates: bool = True):
    """Y = Attn(X W_qkv^T) W_o^T for x [B*N, d_model].

    Returns (y [B*N, d_model], qkv [B*N, (Hq+2Hkv)*d], o [B*N, Hq*d],
    lse [B, Hq, N]); qkv and o as the next step used them.
    """
    w_qkv = np.asarray(w_qkv, dtype=np.float64)
    d = w_qkv.shape[0] // (Hq + 2 * Hkv)
    rnd = round_bf16 if round_intermediates else (lambda a: a)
    qkv = rnd(gemm_nt(x, w_qkv))
    q, k, v = split_heads(qkv, B, N, Hq, Hkv, d)
    o4, lse = attention(q, k, v, causal, scale)
    o = rnd(merge_heads(o4))
    y = gemm_nt(o, w_o)
    return y, qkv, o, lse


def layer_rows(x, w_qkv, w_o, B: int, N: int, Hq: int, Hkv: int, causal: bool, scale: float, b: int, tokens,
               round_intermediates: bool = True):
    """Rows of Y (and of QKV and O) for tokens `tokens` of sequence b only.

    K and V are needed for the whole sequence; Q only for the chosen tokens.
    The same definition as ``layer``, for problems too large to evaluate in
    full.  Returns (y, qkv, o) for those tokens.
    """
    x = np.asarray(x)
    w_qkv = np.asarray(w_qkv, dtype=np.float64)
    d = w_qkv.shape[0] // (Hq + 2 * Hkv)
    rnd = round_bf16 if round_intermediates else (lambda a: a)
    tokens = np.asarray(tokens, dtype=np.int64)
    xs = x[b * N:(b + 1) * N]
    kv = rnd(gemm_nt(xs, w_qkv[Hq * d:]))                      # [N, 2*Hkv*d]
    qkv_t = rnd(gemm_nt(xs[tokens], w_qkv))                    # [T, (Hq+2Hkv)*d]
    o = np.zeros((len(tokens), Hq * d))
    for h in range(Hq):
        g = kv_head_of(h, Hq, Hkv)
        k = kv[:, g * d:(g + 1) * d]
        v = kv[:, (Hkv + g) * d:(Hkv + g + 1) * d]
        o[:, h * d:(h + 1) * d], _ = attention_head(qkv_t[:, h * d:(h + 1) * d], k, v, causal, scale,
                                                    row_index=tokens, n_q=N)
    o = rnd(o)
    return gemm_nt(o, w_o), qkv_t, o
