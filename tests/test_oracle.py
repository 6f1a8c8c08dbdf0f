"""Pins of the fp64 oracle to things other than itself.

Each check below would fail on a plausible slip in oracle/attention_fp64.py: a
dropped or flipped scale, a transposed operand, a wrong mask offset, a wrong
GQA map, a missing normalisation, a wrong LSE base or a wrong combine weight.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import (attention, attention_head, attention_rows, attention_split,
                    combine_partials)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _arr(x):
    return np.array(x, dtype=object).astype(str).astype(np.float64) if _has_str(x) else np.array(x, np.float64)


def _has_str(x):
    if isinstance(x, str):
        return True
    if isinstance(x, list):
        return any(_has_str(e) for e in x)
    return False


def _rng(seed):
    return np.random.default_rng(seed)


def brute_force(q, k, v, causal, scale):
    """Second evaluator, written independently: pure Python, exact sums.

    Uses math.fsum for every reduction and the definition
    p_ij = exp(s_ij) / sum_j exp(s_ij) evaluated with an explicit shift.
    """
    B, Hq, Nq, _ = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    dv = v.shape[3]
    group = Hq // Hkv
    o = np.zeros((B, Hq, Nq, dv))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for i in range(Nq):
                logits = []
                for j in range(Nkv):
                    if causal and j > i + Nkv - Nq:
                        continue
                    dot = math.fsum(float(q[b, h, i, c]) * float(k[b, g, j, c]) for c in range(q.shape[3]))
                    logits.append((j, scale * dot))
                if not logits:
                    lse[b, h, i] = -math.inf
                    continue
                top = max(s for _, s in logits)
                w = [(j, math.exp(s - top)) for j, s in logits]
                z = math.fsum(x for _, x in w)
                for c in range(dv):
                    o[b, h, i, c] = math.fsum(x * float(v[b, g, j, c]) for j, x in w) / z
                lse[b, h, i] = top + math.log(z)
    return o, lse


# ---------------------------------------------------------------- hand cases

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_hand_cases(case):
    q, k, v = (_arr(case[n]) for n in ("q", "k", "v"))
    o, lse = attention(q, k, v, case["causal"], case["scale"])
    np.testing.assert_allclose(o, _arr(case["o"]), rtol=0, atol=1e-14)
    want = _arr(case["lse"])
    assert np.array_equal(np.isinf(lse), np.isinf(want))
    fin = np.isfinite(want)
    np.testing.assert_allclose(lse[fin], want[fin], rtol=0, atol=1e-14)


@pytest.mark.parametrize("case", _golden()["combine_cases"], ids=lambda c: c["name"])
def test_combine_hand_cases(case):
    o, lse = combine_partials(_arr(case["o_parts"]), _arr(case["lse_parts"]))
    np.testing.assert_allclose(o, _arr(case["o"]), rtol=0, atol=1e-14)
    assert abs(lse - case["lse"]) < 1e-14


# ------------------------------------------------------------ closed forms

def test_softmax_rows_sum_to_one_and_mask_is_exact():
    r = _rng(1)
    q = r.standard_normal((37, 16))
    k = r.standard_normal((53, 16))
    v = r.standard_normal((53, 8))
    for causal in (False, True):
        _, _, p = attention_head(q, k, v, causal, 0.3, return_p=True)
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        if causal:
            i = np.arange(37)[:, None]
            j = np.arange(53)[None, :]
            hidden = j > i + (53 - 37)
            assert np.all(p[hidden] == 0.0)
            assert np.all(p[~hidden] > 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_v(causal):
    r = _rng(2)
    n, d, dv = 19, 8, 5
    q = r.standard_normal((1, 1, n, d))
    kk = r.standard_normal(d)
    k = np.tile(kk, (1, 1, n, 1))
    v = r.standard_normal((1, 1, n, dv))
    scale = 0.7
    o, lse = attention(q, k, v, causal, scale)
    for i in range(n):
        seen = i + 1 if causal else n
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :seen].mean(axis=0), rtol=0, atol=1e-13)
        want = scale * float(q[0, 0, i] @ kk) + math.log(seen)
        assert abs(lse[0, 0, i] - want) < 1e-12


def test_causal_row0_selects_v0():
    r = _rng(3)
    q = r.standard_normal((2, 3, 11, 16)) * 4
    k = r.standard_normal((2, 3, 11, 16))
    v = r.standard_normal((2, 3, 11, 7))
    o, lse = attention(q, k, v, True, 0.25)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    s00 = 0.25 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_one_hot_logits_select_one_row(causal):
    d = n = 16
    scale = 0.125
    r = _rng(4)
    perm = r.permutation(n)
    k = 40.0 * np.eye(n, d)[None, None]
    q = (np.eye(d)[perm] / scale)[None, None]
    v = r.standard_normal((1, 1, n, 3))
    o, _ = attention(q, k, v, causal, scale)
    for i in range(n):
        j = perm[i]
        if causal and j > i:
            # The selected key is masked: the row must not select it.
            continue
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, j], rtol=0, atol=1e-15 + 64 * math.exp(-40) * 4)


def test_zero_scale_is_uniform():
    r = _rng(5)
    q = r.standard_normal((1, 2, 9, 4))
    k = r.standard_normal((1, 2, 13, 4))
    v = r.standard_normal((1, 2, 13, 3))
    o, lse = attention(q, k, v, False, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(13), atol=1e-14)


def test_two_keys_closed_form():
    r = _rng(6)
    q = r.standard_normal((1, 1, 5, 3))
    k = r.standard_normal((1, 1, 2, 3))
    v = r.standard_normal((1, 1, 2, 4))
    scale = 1.3
    o, lse = attention(q, k, v, False, scale)
    for i in range(5):
        s0 = scale * q[0, 0, i] @ k[0, 0, 0]
        s1 = scale * q[0, 0, i] @ k[0, 0, 1]
        sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        np.testing.assert_allclose(o[0, 0, i], sig * v[0, 0, 0] + (1 - sig) * v[0, 0, 1], atol=1e-14)
        assert abs(lse[0, 0, i] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-13


def test_single_key():
    q = np.array([[[[0.5, -2.0]]]])
    k = np.array([[[[3.0, 1.0]]]])
    v = np.array([[[[4.0, 5.0, 6.0]]]])
    o, lse = attention(q, k, v, False, 0.5)
    np.testing.assert_array_equal(o[0, 0, 0], [4.0, 5.0, 6.0])
    assert lse[0, 0, 0] == 0.5 * (1.5 - 2.0)


# ------------------------------------------------------------- invariants

def test_permutation_equivariance_noncausal():
    r = _rng(7)
    q = r.standard_normal((1, 1, 8, 6))
    k = r.standard_normal((1, 1, 21, 6))
    v = r.standard_normal((1, 1, 21, 5))
    o1, l1 = attention(q, k, v, False, 0.4)
    perm = r.permutation(21)
    o2, l2 = attention(q, k[:, :, perm], v[:, :, perm], False, 0.4)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_row_shift_changes_lse_not_o(causal):
    # Appending a column a_i to q and a column of ones to k adds scale*a_i to
    # every logit of row i.
    r = _rng(8)
    q = r.standard_normal((1, 1, 10, 4))
    k = r.standard_normal((1, 1, 10, 4))
    v = r.standard_normal((1, 1, 10, 3))
    a = r.standard_normal(10) * 5
    scale = 0.6
    q2 = np.concatenate([q, a[None, None, :, None]], axis=3)
    k2 = np.concatenate([k, np.ones((1, 1, 10, 1))], axis=3)
    o1, l1 = attention(q, k, v, causal, scale)
    o2, l2 = attention(q2, k2, v, causal, scale)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, scale * a[None, None], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_kv(causal):
    r = _rng(9)
    B, Hq, Hkv, N, d = 2, 6, 2, 9, 4
    q = r.standard_normal((B, Hq, N, d))
    k = r.standard_normal((B, Hkv, N, d))
    v = r.standard_normal((B, Hkv, N, 3))
    o1, l1 = attention(q, k, v, causal, 0.5)
    rep = Hq // Hkv
    o2, l2 = attention(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), causal, 0.5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # Head h uses KV head h // 3: swapping KV heads must change head 0 only
    # through its own group.
    o3, _ = attention(q, k[:, ::-1], v[:, ::-1], causal, 0.5)
    assert not np.allclose(o1[:, :3], o3[:, :3])


@pytest.mark.parametrize("causal", [False, True])
def test_split_identity(causal):
    r = _rng(10)
    q = r.standard_normal((2, 2, 7, 5)) * 2
    k = r.standard_normal((2, 2, 29, 5))
    v = r.standard_normal((2, 2, 29, 4))
    o1, l1 = attention(q, k, v, causal, 0.9)
    for bounds in ([0, 29], [0, 10, 29], [0, 1, 2, 15, 28, 29], [0, 23, 26, 29]):
        o2, l2 = attention_split(q, k, v, causal, 0.9, bounds)
        np.testing.assert_allclose(o2, o1, atol=1e-12)
        np.testing.assert_allclose(l2, l1, atol=1e-12)


def test_rows_subset_matches_full():
    r = _rng(11)
    q = r.standard_normal((2, 4, 33, 8))
    k = r.standard_normal((2, 2, 40, 8))
    v = r.standard_normal((2, 2, 40, 6))
    o, lse = attention(q, k, v, True, 0.35)
    rows = [0, 5, 32, 17]
    o2, l2 = attention_rows(q, k, v, True, 0.35, 1, 3, rows)
    np.testing.assert_array_equal(o2, o[1, 3, rows])
    np.testing.assert_array_equal(l2, lse[1, 3, rows])


def test_panels_do_not_change_results(monkeypatch):
    import oracle.attention_fp64 as oa
    r = _rng(12)
    q = r.standard_normal((50, 4))
    k = r.standard_normal((31, 4))
    v = r.standard_normal((31, 2))
    o1, l1 = oa.attention_head(q, k, v, True, 0.5, n_q=50)
    monkeypatch.setattr(oa, "_PANEL_ROWS", 7)
    o2, l2 = oa.attention_head(q, k, v, True, 0.5, n_q=50)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-14)


def test_large_logits_stay_finite():
    r = _rng(13)
    q = r.standard_normal((1, 2, 64, 64)) * 8
    k = r.standard_normal((1, 2, 64, 64))
    v = r.standard_normal((1, 2, 64, 64))
    o, lse = attention(q, k, v, True, 1.0)   # logits of order 60
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


# ------------------------------------------------------- brute force, tiny

@pytest.mark.parametrize("seed,B,Hq,Hkv,Nq,Nkv,d,dv,causal", [
    (20, 1, 1, 1, 1, 1, 3, 2, False),
    (21, 1, 2, 1, 3, 5, 4, 3, True),
    (22, 2, 2, 2, 8, 8, 5, 4, True),
    (23, 1, 4, 2, 6, 8, 8, 8, False),
    (24, 1, 1, 1, 8, 3, 2, 2, True),    # Nq > Nkv: fully masked rows
    (25, 1, 3, 3, 7, 7, 16, 16, False),
])
def test_brute_force_tiny(seed, B, Hq, Hkv, Nq, Nkv, d, dv, causal):
    r = _rng(seed)
    q = r.standard_normal((B, Hq, Nq, d)) * 3
    k = r.standard_normal((B, Hkv, Nkv, d))
    v = r.standard_normal((B, Hkv, Nkv, dv))
    o1, l1 = attention(q, k, v, causal, 0.45)
    o2, l2 = brute_force(q, k, v, causal, 0.45)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    assert np.array_equal(np.isinf(l1), np.isinf(l2))
    fin = np.isfinite(l2)
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_math_fp64(causal):
    # Library cross-check (torch's fp64 math path) for square problems, where
    # torch's top-left causal alignment equals the bottom-right reading.
    r = _rng(30)
    q = r.standard_normal((2, 4, 40, 16))
    k = r.standard_normal((2, 4, 40, 16))
    v = r.standard_normal((2, 4, 40, 8))
    o1, _ = attention(q, k, v, causal, 0.3)
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        is_causal=causal, scale=0.3)
    np.testing.assert_allclose(o1, t.numpy(), rtol=0, atol=1e-12)
