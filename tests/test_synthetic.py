"""Checks of the seeded input generator against published definitions."""
import numpy as np
import torch

from blackwell_programming_gb300 import synthetic as syn


def test_splitmix64_published_vectors():
    # First outputs of SplitMix64 from state 0 (Vigna's reference splitmix64.c).
    z = syn.splitmix64(np.arange(3, dtype=np.uint64), 0)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniform_range_and_moments():
    u = syn.uniform53(np.arange(1 << 20, dtype=np.uint64), 7)
    assert u.min() > 0.0 and u.max() <= 1.0
    assert abs(u.mean() - 0.5) < 2e-3
    assert abs(u.var() - 1.0 / 12.0) < 2e-3


def test_normals_moments_and_chunking():
    x = syn.normals_f32(3, 0, 1 << 20)
    assert x.dtype == np.float32
    assert abs(float(x.mean())) < 5e-3
    assert abs(float(x.std()) - 1.0) < 5e-3
    # Any window of the stream is the same numbers, whatever the chunking.
    y = syn.normals_f32(3, 12345, 1001)
    np.testing.assert_array_equal(x[12345:12345 + 1001], y)
    z = syn.normals_f32(3, 1, 2)
    np.testing.assert_array_equal(x[1:3], z)


def test_bf16_rounding_matches_torch_rne():
    r = np.random.default_rng(0)
    x = np.concatenate([
        r.standard_normal(100000).astype(np.float32) * 10,
        # exact ties: low 16 bits = 0x8000 above even and odd upper halves
        (((np.arange(1000, dtype=np.uint32) + 0x3F80) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38], dtype=np.float32),
    ])
    mine = syn.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


def test_widening_is_exact():
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]        # finite values only
    w = syn.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(w, ref)


def test_workload_inputs_deterministic_and_ordered():
    wl = syn.WORKLOADS["tile_d64"]
    a = syn.make_inputs(wl)
    b = syn.make_inputs(wl)
    np.testing.assert_array_equal(a.q, b.q)
    np.testing.assert_array_equal(a.v, b.v)
    # Q, K, V are consecutive windows of one stream.
    n = 128 * 64
    allx = syn.f32_to_bf16_bits(syn.normals_f32(0, 0, 3 * n))
    np.testing.assert_array_equal(a.q.ravel(), allx[:n])
    np.testing.assert_array_equal(a.k.ravel(), allx[n:2 * n])
    np.testing.assert_array_equal(a.v.ravel(), allx[2 * n:])


def test_q_factor_applied_in_fp32_before_rounding():
    wl = syn.WORKLOADS["causal_d64_bigq"].with_sizes(B=1, Hq=1, Hkv=1, Nq=4, Nkv=4)
    inp = syn.make_inputs(wl)
    raw = syn.normals_f32(0, 0, 4 * 64)
    np.testing.assert_array_equal(inp.q.ravel(), syn.f32_to_bf16_bits(raw * np.float32(8.0)))


def test_flop_and_byte_counts():
    w = syn.WORKLOADS
    assert w["tile_d64"].flops == 4 * 128 * 128 * 64
    assert w["causal_d64_bigq"].flops == 4 * 2 * 8 * 1024 ** 2 * 64 / 2
    assert w["gqa_causal_d128"].flops == 4 * 4 * 32 * 4096 ** 2 * 128 / 2
    assert w["decode_d576"].flops == 2 * 64 * 128 * 8192 * (576 + 512)
    assert w["gqa_causal_d128"].algorithmic_bytes == (
        4 * 32 * 4096 * 128 * 2 + 2 * 4 * 8 * 4096 * 128 * 2 + 4 * 32 * 4096 * 128 * 4 + 4 * 32 * 4096 * 4)
    d = w["decode_d576"]
    assert d.algorithmic_bytes == 64 * 128 * 576 * 2 + 64 * 8192 * 576 * 2 + 64 * 128 * 512 * 4 + 64 * 128 * 4
