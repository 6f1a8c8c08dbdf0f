"""Pins for the layer-slice oracle (QKV projection -> attention -> O projection),
independent of the oracle's own code: exact bf16 ties, a library conversion,
reductions to plain attention under identity-like weights, a pure-Python
brute force, and exact linearity."""
import math

import numpy as np
import pytest
import torch

from oracle import attention, layer, layer_rows, round_bf16


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_ties_and_exact_values():
    # bf16 keeps 8 significant bits: at 1.0 the spacing is 2^-7
    u = 2.0 ** -7
    cases = {
        1.0: 1.0,
        1.0 + u / 2: 1.0,                       # tie -> even (1.0)
        1.0 + 3 * u / 2: 1.0 + 2 * u,           # tie -> even (1 + 2^-6)
        1.0 + u / 2 + 2.0 ** -30: 1.0 + u,      # just past the tie
        1.0 + u / 2 - 2.0 ** -30: 1.0,
        -(1.0 + u / 2 + 2.0 ** -30): -(1.0 + u),
        3.0: 3.0,
        0.0: 0.0,
        2.0 ** -20 * (1 + u): 2.0 ** -20 * (1 + u),
        255.5: 256.0,                           # 255.5 lies between 255 and 256, tie -> 256 (even)
        254.5: 254.0,
    }
    for x, want in cases.items():
        assert round_bf16(x) == want, (x, round_bf16(x), want)


def test_round_bf16_matches_library_on_fp32_values():
    # fp32 inputs have a single rounding to bf16 in torch, so the two agree exactly
    r = np.random.default_rng(3)
    x = (r.standard_normal(200000) * np.exp(r.uniform(-20, 20, 200000))).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(round_bf16(x.astype(np.float64)), lib)


# ------------------------------------------------------------- structure pins

def _bf16_values(r, shape):
    return round_bf16(r.standard_normal(shape))


def test_identity_weights_reduce_to_attention():
    """W_q = I, W_k = a column permutation, W_v = 2 I, W_o = I: the layer is
    plain attention on X cut into heads, built here by explicit loops."""
    B, N, H, d = 2, 5, 2, 4
    D = H * d
    r = np.random.default_rng(11)
    x = _bf16_values(r, (B * N, D))
    perm = r.permutation(D)
    w_q = np.eye(D)
    w_k = np.eye(D)[perm]                     # row j picks feature perm[j]
    w_v = 2.0 * np.eye(D)
    w_qkv = np.concatenate([w_q, w_k, w_v])
    w_o = np.eye(D)
    scale = 0.3
    for causal in (False, True):
        y, qkv, o, lse = layer(x, w_qkv, w_o, B, N, H, H, causal, scale)
        q = np.zeros((B, H, N, d))
        k = np.zeros((B, H, N, d))
        v = np.zeros((B, H, N, d))
        for b in range(B):
            for i in range(N):
                row = x[b * N + i]
                for h in range(H):
                    for c in range(d):
                        q[b, h, i, c] = row[h * d + c]
                        k[b, h, i, c] = row[perm[h * d + c]]
                        v[b, h, i, c] = 2.0 * row[h * d + c]
        o_ref, lse_ref = attention(q, k, v, causal, scale)
        want = np.zeros((B * N, D))
        for b in range(B):
            for i in range(N):
                for h in range(H):
                    want[b * N + i, h * d:(h + 1) * d] = round_bf16(o_ref[b, h, i])
        assert np.array_equal(o, want)
        assert np.array_equal(y, want)
        assert np.array_equal(lse, lse_ref)


def test_grouped_query_slices():
    """Hq = 4 query heads on Hkv = 2 KV heads: K and V come from their own
    column blocks, and query head h reads KV head h // 2."""
    B, N, Hq, Hkv, d = 1, 6, 4, 2, 2
    D = 8
    r = np.random.default_rng(5)
    x = _bf16_values(r, (B * N, D))
    w_q = np.eye(D)                            # Q heads = x columns (0,1), (2,3), ...
    w_k = np.eye(D)[:4]                        # K heads = x columns (0,1) and (2,3)
    w_v = np.eye(D)[4:]                        # V heads = x columns (4,5) and (6,7)
    w_qkv = np.concatenate([w_q, w_k, w_v])
    w_o = np.eye(D)
    y, _, _, _ = layer(x, w_qkv, w_o, B, N, Hq, Hkv, False, 0.7)
    for h in range(Hq):
        g = h // 2
        q = x[:, 2 * h:2 * h + 2][None, None]
        k = x[:, 2 * g:2 * g + 2][None, None]
        v = x[:, 4 + 2 * g:4 + 2 * g + 2][None, None]
        o_ref, _ = attention(q, k, v, False, 0.7)
        assert np.array_equal(y[:, 2 * h:2 * h + 2], round_bf16(o_ref[0, 0]))


def _brute_layer(x, w_qkv, w_o, N, Hq, Hkv, d, causal, scale):
    """The whole slice in pure Python floats, one token at a time."""
    T = len(x)
    nqkv = len(w_qkv)
    qkv = [[sum(x[t][c] * w_qkv[n][c] for c in range(len(x[0]))) for n in range(nqkv)] for t in range(T)]
    o = [[0.0] * (Hq * d) for _ in range(T)]
    for t in range(T):
        b, i = divmod(t, N)
        for h in range(Hq):
            g = h * Hkv // Hq
            q = qkv[t][h * d:(h + 1) * d]
            logits = []
            for j in range(N):
                if causal and j > i:
                    continue
                kj = qkv[b * N + j][(Hq + g) * d:(Hq + g + 1) * d]
                logits.append((j, scale * sum(q[c] * kj[c] for c in range(d))))
            mx = max(s for _, s in logits)
            den = sum(math.exp(s - mx) for _, s in logits)
            for j, s in logits:
                vj = qkv[b * N + j][(Hq + Hkv + g) * d:(Hq + Hkv + g + 1) * d]
                for c in range(d):
                    o[t][h * d + c] += math.exp(s - mx) / den * vj[c]
    return [[sum(o[t][c] * w_o[n][c] for c in range(Hq * d)) for n in range(len(w_o))] for t in range(T)]


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    B, N, D, Hq, Hkv, d = 2, 3, 5, 2, 1, 2
    r = np.random.default_rng(21 + causal)
    x = r.standard_normal((B * N, D))
    w_qkv = r.standard_normal(((Hq + 2 * Hkv) * d, D))
    w_o = r.standard_normal((4, Hq * d))
    y, _, _, _ = layer(x, w_qkv, w_o, B, N, Hq, Hkv, causal, 0.45, round_intermediates=False)
    want = np.array(_brute_layer(x.tolist(), w_qkv.tolist(), w_o.tolist(), N, Hq, Hkv, d, causal, 0.45))
    assert np.max(np.abs(y - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


def test_causal_first_token_closed_form():
    """Token 0 of each sequence sees only itself: its O is its own V."""
    B, N, D, Hq, Hkv, d = 2, 4, 8, 2, 1, 4
    r = np.random.default_rng(9)
    x = _bf16_values(r, (B * N, D))
    w_qkv = _bf16_values(r, ((Hq + 2 * Hkv) * d, D)) / 4
    w_o = _bf16_values(r, (D, Hq * d))
    _, qkv, o, _ = layer(x, w_qkv, w_o, B, N, Hq, Hkv, True, 0.5)
    for b in range(B):
        v0 = qkv[b * N, (Hq + Hkv) * d:]
        for h in range(Hq):
            assert np.array_equal(o[b * N, h * d:(h + 1) * d], round_bf16(v0))


def test_linear_in_output_weight_and_rows_agree():
    B, N, D, Hq, Hkv, d = 2, 7, 16, 4, 2, 4
    r = np.random.default_rng(2)
    x = _bf16_values(r, (B * N, D))
    w_qkv = _bf16_values(r, ((Hq + 2 * Hkv) * d, D)) / 4
    w_o = _bf16_values(r, (D, Hq * d)) / 4
    y, qkv, o, _ = layer(x, w_qkv, w_o, B, N, Hq, Hkv, True, 0.5)
    y2, _, _, _ = layer(x, w_qkv, 2.0 * w_o, B, N, Hq, Hkv, True, 0.5)
    assert np.array_equal(y2, 2.0 * y)                 # a power of two scales exactly
    toks = [0, 3, 6]
    yr, qr, orows = layer_rows(x, w_qkv, w_o, B, N, Hq, Hkv, True, 0.5, 1, toks)
    rows = [N + t for t in toks]
    assert np.allclose(yr, y[rows], rtol=0, atol=1e-12)
    assert np.allclose(qr, qkv[rows], rtol=0, atol=0)
    assert np.allclose(orows, o[rows], rtol=0, atol=1e-15)
