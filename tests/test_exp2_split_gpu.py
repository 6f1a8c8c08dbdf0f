"""The SFU/FMA split of the softmax's exponentials (ATTN_EXP2_SPLIT).

ex2_fma2 evaluates 2^x on the FMA pipe (Cody-Waite reduction to [-1/2, 1/2],
a fitted degree-3 polynomial, the integer part added to the exponent field).
A test-only kernel (tests/cuda/exp2_split.cu) runs it beside the SFU's
ex2.approx; its relative error must stay below 2^-10 (the bf16 rounding of P
that follows is 2^-9) over the arguments the softmax produces, x in
[-125, 8].  The attention path with one exponential pair in four or eight on
the FMA pipe must then meet the same parity bar against the fp64 oracle as
the default path.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("ex2") / "libexp2_split.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-o", out, os.path.join(HERE, "cuda", "exp2_split.cu")], check=True)
    L = ctypes.CDLL(out)
    L.run_exp2_both.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    L.run_exp2_both.restype = ctypes.c_int
    return L


def _both(lib, x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    poly = np.empty_like(x)
    sfu = np.empty_like(x)
    assert lib.run_exp2_both(x.ctypes.data, poly.ctypes.data, sfu.ctypes.data, x.size) == 0
    return poly, sfu


def test_polynomial_against_sfu_exponential(lib):
    rng = np.random.default_rng(3)
    x = np.concatenate([np.linspace(-125.0, 8.0, 400001), rng.uniform(-125.0, 8.0, 200000),
                        rng.uniform(-1.0, 1.0, 100000), np.arange(-125.0, 9.0)]).astype(np.float32)
    poly, sfu = _both(lib, x)
    exact = np.exp2(x.astype(np.float64))
    rel_sfu = np.abs(poly / sfu.astype(np.float64) - 1.0)
    rel_exact = np.abs(poly / exact - 1.0)
    assert rel_sfu.max() <= 2.0 ** -10
    assert rel_exact.max() <= 8e-5          # the fit's own bound, 7.5e-5, plus fp32 rounding
    # integer arguments: the reduction leaves f = 0, so 2^n up to the polynomial's value at 0
    ints = np.arange(-125.0, 9.0, dtype=np.float32)
    p_int, _ = _both(lib, ints)
    assert np.all(np.abs(p_int / np.exp2(ints.astype(np.float64)) - 1.0) <= 8e-5)


def test_arguments_below_range_give_the_floor(lib):
    x = np.array([-125.0, -126.0, -200.0, -1e30, -np.inf], dtype=np.float32)
    poly, _ = _both(lib, x)
    floor = np.exp2(-125.0)
    assert np.all(np.abs(poly / floor - 1.0) <= 8e-5)


@pytest.mark.parametrize("split", ["4", "8"])
@pytest.mark.parametrize("case", [
    ("split_d64_causal_bigq", 2, 4, 4, 700, 700, 64, True, 0.125, 8.0),
    ("split_d128_gqa", 1, 8, 2, 520, 520, 128, True, 128 ** -0.5, 1.0),
    ("split_d128_noncausal_ragged", 2, 4, 1, 300, 455, 128, False, 128 ** -0.5, 1.0),
    ("split_d128_causal_nq_gt_nkv", 1, 2, 2, 300, 170, 128, True, 0.1, 1.0),
])
def test_attention_with_split_matches_oracle(split, case):
    import blackwell_programming_gb300 as gb
    from blackwell_programming_gb300 import synthetic as syn
    from oracle import attention
    from tests.parity_util import check, run_gpu
    gb.build()
    name, B, Hq, Hkv, Nq, Nkv, d, causal, scale, qf = case
    wl = syn.Workload(name, B, Hq, Hkv, Nq, Nkv, d, d, causal, scale, q_factor=qf)
    inp = syn.make_inputs(wl)
    old = os.environ.get("ATTN_EXP2_SPLIT")
    os.environ["ATTN_EXP2_SPLIT"] = split
    try:
        o, lse = run_gpu(inp)
    finally:
        if old is None:
            del os.environ["ATTN_EXP2_SPLIT"]
        else:
            os.environ["ATTN_EXP2_SPLIT"] = old
    q, k, v = inp.f64()
    o_ref, lse_ref = attention(q, k, v, causal, scale)
    check(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, name + " split " + split)
