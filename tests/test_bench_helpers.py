"""bench.py's helpers on the CPU: the sampled parity check that goes into the
bench line (it must accept the oracle's own output and reject a planted
error, with and without dropout) and the roofline object per kernel kind."""
import numpy as np
import pytest

import bench
from blackwell_programming_gb300 import synthetic as syn
from oracle import attention, attention_dropout

torch = pytest.importorskip("torch")


@pytest.fixture
def plain():
    old = bench.DROPOUT
    bench.DROPOUT = 0.0
    yield
    bench.DROPOUT = old


def _wl():
    return syn.Workload("helpers", 2, 4, 2, 70, 90, 64, 64, True, 0.125)


def test_sampled_parity_accepts_the_oracle_and_rejects_a_planted_error(plain):
    wl = _wl()
    inp = syn.make_inputs(wl)
    q, k, v = inp.f64()
    o, lse = attention(q, k, v, wl.causal, wl.scale)
    o_t, l_t = torch.from_numpy(o.astype(np.float32)), torch.from_numpy(lse.astype(np.float32))
    r = bench.sampled_parity(wl, inp, o_t, l_t, heads=8)
    assert r["ok"] and r["max_abs_dO"] < 1e-6 and r["rows"] == 8 * min(48, wl.Nq)
    bad = o_t.clone()
    bad[:, :, :, 3] += 0.05          # every sampled row sees it
    assert not bench.sampled_parity(wl, inp, bad, l_t, heads=8)["ok"]
    bad_l = l_t.clone()
    bad_l += 0.01
    assert not bench.sampled_parity(wl, inp, o_t, bad_l, heads=8)["ok"]


def test_sampled_parity_with_dropout_uses_the_dropout_oracle():
    old = bench.DROPOUT
    bench.DROPOUT = 0.1
    try:
        wl = _wl()
        inp = syn.make_inputs(wl)
        q, k, v = inp.f64()
        o, lse = attention_dropout(q, k, v, wl.causal, wl.scale, 0.1, bench.DROPOUT_SEED)
        r = bench.sampled_parity(wl, inp, torch.from_numpy(o.astype(np.float32)),
                                 torch.from_numpy(lse.astype(np.float32)), heads=8)
        assert r["ok"] and r["max_abs_dO"] < 1e-6
        assert r["bar"]["max_abs_dO"] > bench.O_MAX_ABS      # scaled by the keep factor
        o_plain, _ = attention(q, k, v, wl.causal, wl.scale)
        r = bench.sampled_parity(wl, inp, torch.from_numpy(o_plain.astype(np.float32)),
                                 torch.from_numpy(lse.astype(np.float32)), heads=8)
        assert r["max_abs_dO"] > 1e-3                       # the dropout-free O is not the answer
    finally:
        bench.DROPOUT = old


def test_roofline_kinds(plain):
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0}
    roof, kind = bench.roofline_for(syn.WORKLOADS["gqa_causal_d128"], 0.5e-3, peaks, "test")
    assert kind == "prefill" and roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["achieved"] == pytest.approx(syn.WORKLOADS["gqa_causal_d128"].flops / 0.5e-3 / 1e12)
    assert roof["frac"] == pytest.approx(roof["achieved"] / 1800.0)
    roof, kind = bench.roofline_for(syn.WORKLOADS["decode_d576"], 0.2e-3, peaks, "test")
    assert kind == "decode" and roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] == pytest.approx(syn.WORKLOADS["decode_d576"].algorithmic_bytes / 0.2e-3 / 1e9)
    roof, kind = bench.roofline_for(syn.WORKLOADS["mla_prefill_causal"], 1e-3, peaks, "test")
    assert kind == "latent_prefill" and roof["bound"] == "tensor"
