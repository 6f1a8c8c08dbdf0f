"""fp64 CPU oracle for the fused attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` call it.  It shares no code with the CUDA path.

What it computes is the plain definition of attention written out, with the
full score matrix materialised:

    O = softmax(mask(scale * Q K^T)) V

in the stage order of the FlashAttention pipeline drawn on "CS149 L11:
Programming Specialized Hardware" (section 5, the FlashAttention-as-a-
metapipeline slide: QK^T -> Mask -> Softmax -> x V; dropout is not part of an
inference forward and is left out), with the softmax done as the three
parallel patterns of the simplified-softmax slide of the same section:
Map (exp), Reduce (+), Zip (/).

The tiled GPU kernel reaches the same numbers through an online softmax (the
running max and normaliser of the FA2-style kernel in "Distilling a 4.5 hour
CUDA talk", section 7) and base-2 exponentials with log2(e) folded into the
scale (same page, sections 2 and 7).  Both are exact rewrites of this
definition up to rounding, so the oracle does not follow them: it subtracts
the row maximum (exact in the mathematics, it only keeps fp64 in range) and
uses the natural exponential.

Readings where the pages are silent:
* LSE is the natural log of sum_j exp(scale * q_i . k_j) over unmasked keys.
* Causal masking is aligned bottom-right: key j is visible to query i iff
  j <= i + (Nkv - Nq).
* A row with no visible key has O = 0 and LSE = -inf.
* Grouped-query attention maps query head h to KV head h // (Hq // Hkv).
* Split-KV partials (O_s, lse_s) over a partition of the keys combine as
  LSE = log sum_s exp(lse_s),  O = sum_s exp(lse_s - LSE) O_s.

Every function here is pinned by tests/test_oracle.py against closed forms,
invariants, hand-derived cases and an independent brute-force evaluator.
"""
from __future__ import annotations

import numpy as np

# Rows of the score matrix materialised at once.  Rows are independent, so the
# panel size changes memory use and (through the matmul library's blocking)
# the last bits of rounding only.
_PANEL_ROWS = 2048


def attention_head(q, k, v, causal: bool, scale: float, row_index=None, n_q=None,
                   key_offset: int = 0, n_kv_total=None, return_p: bool = False):
    """Attention for one (batch, query head) pair in fp64.

    q: [R, d_qk] query rows; k: [n, d_qk]; v: [n, d_v].
    row_index: the position of each q row in its sequence (default 0..R-1),
    and n_q the sequence's query count (default R).  key_offset is the
    position of k[0] in its sequence and n_kv_total the sequence's key count
    (default key_offset + n).  Positions only matter for the causal mask.
    Returns (o [R, d_v], lse [R]) and P [R, n] if asked.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R = q.shape[0]
    n = k.shape[0]
    if row_index is None:
        row_index = np.arange(R)
    row_index = np.asarray(row_index, dtype=np.int64)
    if n_q is None:
        n_q = R
    if n_kv_total is None:
        n_kv_total = key_offset + n

    o = np.zeros((R, v.shape[1]), dtype=np.float64)
    lse = np.full(R, -np.inf, dtype=np.float64)
    p_all = np.zeros((R, n), dtype=np.float64) if return_p else None
    key_pos = key_offset + np.arange(n)

    for r0 in range(0, R, _PANEL_ROWS):
        r1 = min(R, r0 + _PANEL_ROWS)
        # QK^T, scaled.
        s = scale * (q[r0:r1] @ k.T)
        # Mask: key j is hidden from query i when j > i + (Nkv - Nq).
        if causal:
            limit = row_index[r0:r1, None] + (n_kv_total - n_q)
            s = np.where(key_pos[None, :] > limit, -np.inf, s)
        m = s.max(axis=1) if n > 0 else np.full(r1 - r0, -np.inf)
        live = np.isfinite(m)
        # Softmax: Map exp, Reduce +, Zip /.
        e = np.zeros_like(s)
        e[live] = np.exp(s[live] - m[live, None])
        l = e.sum(axis=1)
        p = np.zeros_like(s)
        p[live] = e[live] / l[live, None]
        # x V
        o[r0:r1] = p @ v
        lse_panel = np.full(r1 - r0, -np.inf)
        lse_panel[live] = m[live] + np.log(l[live])
        lse[r0:r1] = lse_panel
        if return_p:
            p_all[r0:r1] = p
    if return_p:
        return o, lse, p_all
    return o, lse


def kv_head_of(h: int, Hq: int, Hkv: int) -> int:
    """Grouped-query map: consecutive groups of Hq // Hkv query heads share a KV head."""
    return h // (Hq // Hkv)


def attention(q, k, v, causal: bool, scale: float):
    """Full attention forward over [B, H, N, d] fp64 arrays.

    q: [B, Hq, Nq, d_qk], k: [B, Hkv, Nkv, d_qk], v: [B, Hkv, Nkv, d_v].
    Returns o [B, Hq, Nq, d_v] and lse [B, Hq, Nq] (fp64).
    """
    B, Hq, Nq, _ = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    o = np.zeros((B, Hq, Nq, v.shape[3]), dtype=np.float64)
    lse = np.zeros((B, Hq, Nq), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            kv = kv_head_of(h, Hq, Hkv)
            o[b, h], lse[b, h] = attention_head(q[b, h], k[b, kv], v[b, kv], causal, scale)
    return o, lse


def attention_rows(q, k, v, causal: bool, scale: float, b: int, h: int, rows):
    """O and LSE of selected query rows of head (b, h) only.

    Same definition as ``attention``; used to check outputs of problems too
    large to evaluate in full.
    """
    Hq = q.shape[1]
    Hkv = k.shape[1]
    kv = kv_head_of(h, Hq, Hkv)
    rows = np.asarray(rows, dtype=np.int64)
    return attention_head(q[b, h, rows], k[b, kv], v[b, kv], causal, scale,
                          row_index=rows, n_q=q.shape[2])


def combine_partials(o_parts, lse_parts):
    """Merge split-KV partials over a partition of the keys.

    o_parts: [S, ..., d_v] normalised partial outputs; lse_parts: [S, ...]
    partial log-sum-exps (natural log).  A partial whose lse is -inf (no
    visible key) contributes nothing; if all are -inf the result is O = 0,
    LSE = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    mx = lse_parts.max(axis=0)
    live = np.isfinite(mx)
    safe = np.where(live, mx, 0.0)
    w = np.exp(lse_parts - safe[None])          # exp(-inf) = 0 for empty parts
    tot = w.sum(axis=0)
    lse = np.where(live, safe + np.log(np.where(live, tot, 1.0)), -np.inf)
    coef = np.where(live[None], w / np.where(live, tot, 1.0)[None], 0.0)
    o = (coef[..., None] * o_parts).sum(axis=0)
    return o, lse


def attention_split(q, k, v, causal: bool, scale: float, bounds):
    """Split-KV evaluation: attention over each key range, then combine.

    bounds: increasing key offsets [0 = b0 < b1 < ... < bS = Nkv].  Each part
    sees keys [b_s, b_{s+1}) under the same (absolute-position) mask as the
    unsplit problem.
    """
    B, Hq, Nq, _ = q.shape
    Hkv = k.shape[1]
    n_kv = k.shape[2]
    parts_o, parts_l = [], []
    for s in range(len(bounds) - 1):
        k0, k1 = bounds[s], bounds[s + 1]
        o_s = np.zeros((B, Hq, Nq, v.shape[3]))
        l_s = np.full((B, Hq, Nq), -np.inf)
        for b in range(B):
            for h in range(Hq):
                kv = kv_head_of(h, Hq, Hkv)
                o_s[b, h], l_s[b, h] = attention_head(
                    q[b, h], k[b, kv, k0:k1], v[b, kv, k0:k1], causal, scale,
                    key_offset=k0, n_kv_total=n_kv)
        parts_o.append(o_s)
        parts_l.append(l_s)
    return combine_partials(np.stack(parts_o), np.stack(parts_l))
