"""fp64 CPU oracle for the attention forward with dropout on the softmax
weights.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
the tests and the CPU-baseline leg of ``bench.py`` call it.  It shares no
code with the CUDA path.

What it computes: the FlashAttention pipeline drawn on "CS149 L11:
Programming Specialized Hardware" (section 5, the metapipeline slide: QK^T,
Mask, Softmax, Dropout, x V), with the dropout stage in place:

    P = softmax(mask(scale * Q K^T))              (as attention_fp64)
    O = (P * Keep) V / keep_probability
    LSE = the log-sum-exp of the masked, scaled logits (dropout does not
          change it)

Readings where the pages are silent (the slide names the stage only):
* Each weight p_ij is dropped independently with probability p, and the kept
  ones are divided by the keep probability, so that the expectation of O over
  the random bits is the dropout-free O (inverted dropout).
* The random bits come from a counter-based generator, Philox4x32-10
  (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
  SC 2011), so any element's bits can be drawn on their own.  For key j of
  query row i (its position in the sequence) in head h of batch b, with a
  64-bit seed: counter (j >> 4, i, h, b), key (seed mod 2^32, seed >> 32);
  the element's 8-bit uniform is byte (j & 3) (the least significant for
  j & 3 = 0) of output word ((j >> 2) & 3), so one call serves 16 keys.
* The probability is quantised to 8 bits: t = floor(p * 256 + 1/2); the
  element is dropped iff its uniform is below t, so the realised drop
  probability is t / 256, and kept weights are scaled by 256 / (256 - t),
  which keeps the expectation exact.

Pinned by tests/test_oracle_dropout.py: p = 0 is plain attention, the
generator's output bits are balanced and every input bit avalanches, the drop
rate and the expectation of O match their targets within binomial and
central-limit bounds, masks do not depend on the problem's size, and a
scalar pure-Python evaluator agrees.  The key schedule's Weyl constants equal
their closed forms (the golden ratio's fractional part and sqrt(3) - 1 in
32-bit fixed point), and an inverse written from the round definition
recovers every counter, which fixes the round structure, the word order and
the round count.  The published known-answer vectors of Philox4x32-10 (the
Random123 library's, tests/golden/philox4x32_10_kat.json) fix the two round
multipliers and the whole output.
"""
from __future__ import annotations

import numpy as np

from .attention_fp64 import attention_head, kv_head_of

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """Philox4x32-10 on arrays: ctr [..., 4] (uint32 values), key (k0, k1).

    Ten rounds.  A round multiplies counter words 0 and 2 by M0 and M1 into
    64-bit products and forms (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2),
    hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)); the key then advances by (W0, W1)
    modulo 2^32.  Returns the [..., 4] output words as uint32.
    """
    c = np.asarray(ctr, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for _ in range(10):
        p0 = np.uint64(PHILOX_M0) * c0
        p1 = np.uint64(PHILOX_M1) * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ np.uint64(k0), p1 & _MASK32,
                          (p0 >> np.uint64(32)) ^ c3 ^ np.uint64(k1), p0 & _MASK32)
        k0 = (k0 + PHILOX_W0) & 0xFFFFFFFF
        k1 = (k1 + PHILOX_W1) & 0xFFFFFFFF
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


KEEP_LEVELS = 256   # the uniforms have 8 bits


def drop_threshold(p: float) -> int:
    """The 8-bit threshold t for drop probability p (0 <= p < 1), computed
    from p as a float32 value, as a C caller passes it."""
    p32 = float(np.float32(p))
    if not 0.0 <= p32 < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    t = int(np.floor(p32 * KEEP_LEVELS + 0.5))
    if t >= KEEP_LEVELS:
        raise ValueError("dropout probability rounds to dropping every weight")
    return t


def keep_scale(t: int) -> float:
    """Factor on kept weights: the inverse of the realised keep probability."""
    return KEEP_LEVELS / (KEEP_LEVELS - t)


def uniforms8(b: int, h: int, rows, n_keys: int, seed: int) -> np.ndarray:
    """The 8-bit uniforms [len(rows), n_keys] of keys 0..n_keys-1 of the given
    query rows of head h in batch b."""
    rows = np.asarray(rows, dtype=np.int64)
    blocks = (n_keys + 15) // 16
    ctr = np.zeros((len(rows), blocks, 4), dtype=np.uint64)
    ctr[..., 0] = np.arange(blocks)[None, :]
    ctr[..., 1] = rows[:, None]
    ctr[..., 2] = h
    ctr[..., 3] = b
    words = philox4x32_10(ctr, (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))   # [R, blocks, 4]
    by = np.stack([(words >> np.uint32(8 * i)) & np.uint32(0xFF) for i in range(4)], axis=-1)
    u = by.reshape(len(rows), blocks * 16)   # key 16*blk + 4*word + byte
    return u[:, :n_keys]


def keep_mask(b: int, h: int, rows, n_keys: int, seed: int, t: int) -> np.ndarray:
    """True where the weight of (row, key) is kept."""
    return uniforms8(b, h, rows, n_keys, seed) >= t


def attention_dropout_head(q, k, v, causal: bool, scale: float, p_drop: float, seed: int, b: int, h: int,
                           row_index=None, n_q=None):
    """One (batch, query head) pair: O with dropout, and the LSE.

    q [R, d], k [n, d], v [n, d_v]; row_index = positions of the q rows
    (default 0..R-1), n_q = the sequence's query count (default R).
    """
    R = np.asarray(q).shape[0]
    n = np.asarray(k).shape[0]
    if row_index is None:
        row_index = np.arange(R)
    _, lse, p = attention_head(q, k, v, causal, scale, row_index=row_index, n_q=n_q, return_p=True)
    t = drop_threshold(p_drop)
    keep = keep_mask(b, h, row_index, n, seed, t)
    o = (np.where(keep, p, 0.0) @ np.asarray(v, dtype=np.float64)) * keep_scale(t)
    return o, lse


def attention_dropout(q, k, v, causal: bool, scale: float, p_drop: float, seed: int):
    """Dropout attention over [B, H, N, d] arrays; returns o [B, Hq, Nq, d_v], lse [B, Hq, Nq]."""
    B, Hq, Nq, _ = q.shape
    Hkv = k.shape[1]
    o = np.zeros((B, Hq, Nq, v.shape[3]))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            o[b, h], lse[b, h] = attention_dropout_head(q[b, h], k[b, g], v[b, g], causal, scale, p_drop, seed,
                                                        b, h)
    return o, lse


def attention_dropout_rows(q, k, v, causal: bool, scale: float, p_drop: float, seed: int, b: int, h: int, rows):
    """Selected query rows of head (b, h) only, for problems too large to evaluate in full."""
    Hq, Hkv, Nq = q.shape[1], k.shape[1], q.shape[2]
    g = kv_head_of(h, Hq, Hkv)
    rows = np.asarray(rows, dtype=np.int64)
    return attention_dropout_head(q[b, h, rows], k[b, g], v[b, g], causal, scale, p_drop, seed, b, h,
                                  row_index=rows, n_q=Nq)
