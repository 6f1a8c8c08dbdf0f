"""Pins for the dropout oracle and its counter-based generator, independent of
the oracle's own code: the dropout-free special case, statistical properties
of the generator's bits (balance, avalanche), the drop rate and the
expectation of O within binomial / central-limit bounds, size independence of
the masks, and a scalar pure-Python evaluator."""
import math

import numpy as np
import pytest

from oracle import attention
from oracle.dropout_fp64 import (attention_dropout, drop_threshold, keep_mask, keep_scale, philox4x32_10,
                                 uniforms8)


def _inputs(r, B, Hq, Hkv, Nq, Nkv, d):
    q = r.standard_normal((B, Hq, Nq, d))
    k = r.standard_normal((B, Hkv, Nkv, d))
    v = r.standard_normal((B, Hkv, Nkv, d))
    return q, k, v


def test_zero_probability_is_plain_attention():
    r = np.random.default_rng(1)
    q, k, v = _inputs(r, 2, 4, 2, 9, 13, 8)
    for causal in (False, True):
        o, lse = attention_dropout(q, k, v, causal, 0.4, 0.0, seed=1234)
        o_ref, lse_ref = attention(q, k, v, causal, 0.4)
        assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)


def test_threshold_quantisation():
    assert drop_threshold(0.0) == 0
    assert drop_threshold(0.5) == 128
    assert drop_threshold(0.25) == 64
    assert drop_threshold(1.0 / 256) == 1
    assert drop_threshold(0.1) == 26                   # 25.6 rounds up
    assert drop_threshold(0.001) == 0                  # below half a level: nothing is dropped
    assert keep_scale(26) == 256 / 230
    with pytest.raises(ValueError):
        drop_threshold(1.0)
    with pytest.raises(ValueError):
        drop_threshold(0.999)                          # below 1, but t would be 256


def _bits(words):
    return np.unpackbits(np.ascontiguousarray(words).view(np.uint8), axis=-1)


def test_generator_bits_balanced_and_uniform():
    n = 1 << 18
    ctr = np.zeros((n, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(n)
    out = philox4x32_10(ctr, (0x12345678, 0x9ABCDEF0))
    bits = _bits(out)                                  # [n, 128]
    freq = bits.mean(axis=0)
    sigma = 0.5 / math.sqrt(n)
    assert np.all(np.abs(freq - 0.5) < 6 * sigma)
    # every byte: 256 bins, chi-square with 255 degrees of freedom
    u = np.concatenate([((out >> (8 * i)) & 0xFF).ravel() for i in range(4)])
    counts = np.bincount(u, minlength=256)
    e = len(u) / 256
    chi2 = float(((counts - e) ** 2 / e).sum())
    assert 180 < chi2 < 340                            # about +-4.5 sigma around 255


def test_generator_avalanche():
    """Flipping any one bit of the counter or of the key flips half of the 128
    output bits on average (a generator with too few or broken rounds fails)."""
    r = np.random.default_rng(5)
    n = 2048
    base = r.integers(0, 1 << 32, size=(n, 4), dtype=np.uint64)
    key = (0xDEADBEEF, 0x01234567)
    ref = _bits(philox4x32_10(base, key))
    for word in range(4):
        for bit in range(32):
            flipped = base.copy()
            flipped[:, word] ^= np.uint64(1 << bit)
            diff = (_bits(philox4x32_10(flipped, key)) != ref).sum(axis=1).mean()
            assert 62.0 < diff < 66.0, (word, bit, diff)
    for kw in range(2):
        for bit in (0, 7, 31):
            k2 = list(key)
            k2[kw] ^= 1 << bit
            diff = (_bits(philox4x32_10(base, tuple(k2))) != ref).sum(axis=1).mean()
            assert 62.0 < diff < 66.0


def test_drop_rate_binomial():
    for p in (0.1, 0.5, 0.9):
        t = drop_threshold(p)
        keep = keep_mask(1, 3, np.arange(1000), 1000, seed=77, t=t)
        n = keep.size
        q = t / 256.0
        dropped = n - int(keep.sum())
        assert abs(dropped - n * q) < 6 * math.sqrt(n * q * (1 - q))


def test_masks_depend_only_on_position():
    t = drop_threshold(0.3)
    a = keep_mask(0, 2, np.arange(40), 100, seed=9, t=t)
    b = keep_mask(0, 2, np.arange(10, 50), 333, seed=9, t=t)
    assert np.array_equal(a[10:40], b[:30, :100])
    # distinct rows, heads, batches and seeds draw distinct bits
    base = uniforms8(0, 0, [5], 256, seed=1)
    for other in (uniforms8(0, 0, [6], 256, 1), uniforms8(0, 1, [5], 256, 1),
                  uniforms8(1, 0, [5], 256, 1), uniforms8(0, 0, [5], 256, 2),
                  uniforms8(0, 0, [5], 256, 1 << 32)):
        assert not np.array_equal(base, other)


def test_expectation_is_dropout_free_output():
    """Inverted dropout: averaged over seeds, O tends to the dropout-free O
    (a missing or wrong rescale fails this by far)."""
    r = np.random.default_rng(3)
    q, k, v = _inputs(r, 1, 1, 1, 3, 24, 4)
    o_ref, _ = attention(q, k, v, False, 0.5)
    samples = np.stack([attention_dropout(q, k, v, False, 0.5, 0.4, seed=s)[0] for s in range(3000)])
    mean = samples.mean(axis=0)
    sem = samples.std(axis=0) / math.sqrt(len(samples))
    assert np.all(np.abs(mean - o_ref) < 5 * sem + 1e-12)


def _philox_scalar(c, k):
    """Philox4x32-10 in plain integers, one counter at a time."""
    c = [x & 0xFFFFFFFF for x in c]
    k0, k1 = k
    for _ in range(10):
        a = 0xD2511F53 * c[0]
        z = 0xCD9E8D57 * c[2]
        c = [((z >> 32) ^ c[1] ^ k0) & 0xFFFFFFFF, z & 0xFFFFFFFF, ((a >> 32) ^ c[3] ^ k1) & 0xFFFFFFFF,
             a & 0xFFFFFFFF]
        k0 = (k0 + 0x9E3779B9) & 0xFFFFFFFF
        k1 = (k1 + 0xBB67AE85) & 0xFFFFFFFF
    return c


@pytest.mark.parametrize("causal", [False, True])
def test_scalar_evaluator(causal):
    B, Hq, Hkv, Nq, Nkv, d = 1, 2, 1, 5, 11, 3
    r = np.random.default_rng(8 + causal)
    q, k, v = _inputs(r, B, Hq, Hkv, Nq, Nkv, d)
    p_drop, seed, scale = 0.35, (7 << 32) | 99, 0.6
    o, _ = attention_dropout(q, k, v, causal, scale, p_drop, seed)
    t = math.floor(float(np.float32(p_drop)) * 256 + 0.5)
    for h in range(Hq):
        for i in range(Nq):
            logits = {}
            for j in range(Nkv):
                if causal and j > i + Nkv - Nq:
                    continue
                logits[j] = scale * sum(q[0, h, i, c] * k[0, 0, j, c] for c in range(d))
            mx = max(logits.values())
            den = sum(math.exp(s - mx) for s in logits.values())
            want = [0.0] * d
            for j, s in logits.items():
                word = _philox_scalar([j // 16, i, h, 0], (seed & 0xFFFFFFFF, seed >> 32))[(j % 16) // 4]
                u = (word >> (8 * (j % 4))) & 0xFF
                if u < t:
                    continue
                for c in range(d):
                    want[c] += math.exp(s - mx) / den * v[0, 0, j, c] * 256 / (256 - t)
            assert np.max(np.abs(o[0, h, i] - np.array(want))) < 1e-12


def test_weyl_constants_closed_form():
    """The key schedule's increments are the published Weyl constants: the
    golden ratio's fractional part and sqrt(3) - 1, in 32-bit fixed point
    (exact integer square roots, no floating point)."""
    from oracle import dropout_fp64 as dr
    assert dr.PHILOX_W0 == (math.isqrt(5 << 64) - (1 << 32)) // 2
    assert dr.PHILOX_W1 == math.isqrt(3 << 64) - (1 << 32)
    # the round multipliers must be odd, or the round would not be a bijection
    assert dr.PHILOX_M0 & 1 and dr.PHILOX_M1 & 1


def _philox_inverse(out, key, m0, m1, w0, w1, rounds=10):
    """Undo the rounds from the last one back: lo(M * x) gives x through the
    inverse of the odd multiplier modulo 2^32, hi(M * x) then unmasks the
    word that was XORed with it."""
    m0i, m1i = pow(m0, -1, 1 << 32), pow(m1, -1, 1 << 32)
    keys = [((key[0] + r * w0) & 0xFFFFFFFF, (key[1] + r * w1) & 0xFFFFFFFF) for r in range(rounds)]
    y0, y1, y2, y3 = out
    for k0, k1 in reversed(keys):
        x2 = (y1 * m1i) & 0xFFFFFFFF
        x0 = (y3 * m0i) & 0xFFFFFFFF
        x1 = y0 ^ ((m1 * x2) >> 32) ^ k0
        x3 = y2 ^ ((m0 * x0) >> 32) ^ k1
        y0, y1, y2, y3 = x0, x1, x2, x3
    return [y0, y1, y2, y3]


def test_rounds_invert_to_the_counter():
    """Each round is a bijection of the counter for a fixed key.  An inverse
    written from the round's definition must recover every counter from the
    oracle's output: a swapped output word, a hi/lo mix-up, a wrong round
    count or a key schedule that advances before the first round all break
    the round trip."""
    from oracle import dropout_fp64 as dr
    r = np.random.default_rng(11)
    ctr = r.integers(0, 1 << 32, size=(64, 4), dtype=np.uint64)
    key = (0x0BADC0DE, 0xFEEDFACE)
    out = philox4x32_10(ctr, key)
    for c, o in zip(ctr.tolist(), out.tolist()):
        back = _philox_inverse(o, key, dr.PHILOX_M0, dr.PHILOX_M1, dr.PHILOX_W0, dr.PHILOX_W1)
        assert back == c
    # nine or eleven rounds do not invert it
    o = out[0].tolist()
    for rounds in (9, 11):
        assert _philox_inverse(o, key, dr.PHILOX_M0, dr.PHILOX_M1, dr.PHILOX_W0, dr.PHILOX_W1, rounds) != ctr[0].tolist()


def test_published_known_answer_vectors():
    """The generator against the known-answer vectors that the Random123
    library publishes for Philox4x32-10 (Salmon et al., SC 2011): all-zero
    counter and key, all-ones, and the digits-of-pi case.  They fix the two
    round multipliers, which the statistical pins above leave open."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")) as f:
        kat = json.load(f)
    assert len(kat["cases"]) == 3
    for case in kat["cases"]:
        ctr = np.array([int(w, 16) for w in case["counter"]], dtype=np.uint64)
        key = [int(w, 16) for w in case["key"]]
        want = [int(w, 16) for w in case["output"]]
        got = philox4x32_10(ctr, key)
        assert [int(x) for x in got] == want, case
