"""GPU parity of attention with dropout (attn_fwd_dropout) against the fp64
dropout oracle.

* The keep mask is compared bit for bit: with V one-hot over a block of d
  keys (V[j, c] = 1 iff j = j0 + c), O[i, c] is the kept, rescaled weight of
  key j0 + c, which is zero exactly when the kernel dropped it (the weights
  themselves stay far above bf16's smallest normal).
* O with random V meets the attention bar scaled by the dropout factor
  256 / (256 - t): the kernel's errors (bf16 P, fp32 sums) scale with the
  weights it sums, and the kept ones are multiplied by that factor.
* LSE is the dropout-free LSE: bit for bit attn_fwd's.
"""
import numpy as np
import pytest

from blackwell_programming_gb300 import synthetic as syn
from oracle import attention_dropout, attention_dropout_rows, drop_threshold, keep_mask
from oracle.dropout_fp64 import keep_scale
from parity_util import LSE_REL, O_MAX_ABS, O_MEAN_ABS

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SEED = 0x0123456789ABCDEF


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blackwell_programming_gb300 as gbmod
    gbmod.build()
    return gbmod


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def status_ok(gb):
    torch.cuda.synchronize()
    st = gb.attn_check_device(reset=True)
    assert st == 0, "device status %d: %s" % (st, gb.attn_last_cuda_error())


@pytest.mark.parametrize("d,causal", [(128, True), (128, False), (64, True)])
def test_keep_mask_bit_exact(gb, d, causal):
    B, Hq, Hkv, N = 2, 4, 2, 300
    wl = syn.Workload("mask", B, Hq, Hkv, N, N, d, d, causal, 0.05, seed=d + causal)
    inp = syn.make_inputs(wl)
    q, k = to_dev(inp.q), to_dev(inp.k)
    p_drop = 0.3
    t = drop_threshold(p_drop)
    rows = np.arange(N)
    for j0 in range(0, N, d):
        onehot = np.zeros((B, Hkv, N, d), dtype=np.float32)
        for c in range(min(d, N - j0)):
            onehot[:, :, j0 + c, c] = 1.0
        v = torch.from_numpy(onehot).to(torch.bfloat16).cuda()
        gb.attn_check_device(reset=True)
        o, _ = gb.attn_fwd_dropout(q, k, v, p_drop, SEED, causal=causal, scale=wl.scale)
        status_ok(gb)
        o = o.cpu().numpy()
        width = min(d, N - j0)
        keys = j0 + np.arange(width)
        visible = (keys[None, :] <= rows[:, None]) if causal else np.ones((N, width), dtype=bool)
        for b in range(B):
            for h in range(Hq):
                keep = keep_mask(b, h, rows, N, SEED, t)[:, j0:j0 + width]
                got_kept = o[b, h, :, :width] != 0.0
                assert np.array_equal(got_kept, keep & visible), (b, h, j0)


CASES = [
    # B, Hq, Hkv, Nq, Nkv, d, causal, p
    (1, 2, 2, 128, 128, 64, False, 0.1),
    (2, 4, 2, 300, 300, 128, True, 0.1),
    (1, 8, 2, 333, 333, 64, True, 0.5),
    (2, 4, 1, 100, 260, 128, True, 0.25),    # Nq < Nkv
    (1, 4, 4, 513, 513, 128, False, 0.5),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_H%d_%d_N%d_%d_d%d_%s_p%g" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full", c[7]))
def test_dropout_parity(gb, case):
    B, Hq, Hkv, Nq, Nkv, d, causal, p_drop = case
    wl = syn.Workload("drop", B, Hq, Hkv, Nq, Nkv, d, d, causal, 1.0 / np.sqrt(d), seed=sum(case[:6]))
    inp = syn.make_inputs(wl)
    q, k, v = (to_dev(x) for x in (inp.q, inp.k, inp.v))
    gb.attn_check_device(reset=True)
    o, lse = gb.attn_fwd_dropout(q, k, v, p_drop, SEED, causal=causal, scale=wl.scale)
    o0, lse0 = gb.attn_fwd(q, k, v, causal=causal, scale=wl.scale)
    o_again, _ = gb.attn_fwd_dropout(q, k, v, p_drop, SEED, causal=causal, scale=wl.scale)
    o_other, _ = gb.attn_fwd_dropout(q, k, v, p_drop, SEED + 1, causal=causal, scale=wl.scale)
    o_zero, lse_zero = gb.attn_fwd_dropout(q, k, v, 0.0, SEED, causal=causal, scale=wl.scale)
    status_ok(gb)
    assert torch.equal(lse, lse0), "dropout changed the LSE"
    assert torch.equal(o, o_again), "same seed, different result"
    assert not torch.equal(o, o_other), "another seed drew the same mask"
    assert torch.equal(o_zero, o0) and torch.equal(lse_zero, lse0), "p = 0 differs from attn_fwd"
    q64, k64, v64 = inp.f64()
    o_or, lse_or = attention_dropout(q64, k64, v64, causal, wl.scale, p_drop, SEED)
    t = drop_threshold(p_drop)
    f = keep_scale(t)
    err = np.abs(o.cpu().numpy() - o_or)
    assert float(err.max()) <= O_MAX_ABS * f, "max |dO| %.3e" % err.max()
    assert float(err.mean()) <= O_MEAN_ABS * f, "mean |dO| %.3e" % err.mean()
    fin = np.isfinite(lse_or)
    le = np.abs(lse.cpu().numpy()[fin] - lse_or[fin]) / np.maximum(1.0, np.abs(lse_or[fin]))
    assert float(le.max()) <= LSE_REL


def test_dropout_full_size_sampled(gb):
    """The benchmarked GQA causal d=128 workload (4 x 32 heads x 4096) with
    p = 0.1: sampled rows against the oracle."""
    wl = syn.WORKLOADS["gqa_causal_d128"]
    inp = syn.make_inputs(wl)
    q, k, v = (to_dev(x) for x in (inp.q, inp.k, inp.v))
    gb.attn_check_device(reset=True)
    o, lse = gb.attn_fwd_dropout(q, k, v, 0.1, SEED, causal=True, scale=wl.scale)
    _, lse0 = gb.attn_fwd(q, k, v, causal=True, scale=wl.scale)
    status_ok(gb)
    assert torch.equal(lse, lse0)
    q64, k64, v64 = inp.f64()
    f = keep_scale(drop_threshold(0.1))
    rows = [0, 1, 127, 128, 255, 2047, 3000, 4095]
    for b, h in ((0, 0), (3, 31), (1, 17)):
        o_or, _ = attention_dropout_rows(q64, k64, v64, True, wl.scale, 0.1, SEED, b, h, rows)
        err = np.abs(o[b, h, rows].cpu().numpy() - o_or)
        assert float(err.max()) <= O_MAX_ABS * f and float(err.mean()) <= O_MEAN_ABS * f, (b, h, err.max())
