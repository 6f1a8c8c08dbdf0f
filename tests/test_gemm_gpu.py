"""GPU parity of the projection GEMM (gemm_bf16_nt) against the fp64 oracle.

Tolerance, derived from the arithmetic: with bf16 inputs (exact in fp32) the
kernel forms each C[m, n] as an fp32 sum of K exact products in some order,
so |C_gpu - C| <= K * 2^-24 * (|A| |B|^T)[m, n] (the worst-case bound of a
K-term floating-point sum).  bf16 output is that fp32 value rounded once, to
nearest even, and must equal the fp32 output rounded to bf16 bit for bit.
"""
import numpy as np
import pytest

from blackwell_programming_gb300 import synthetic as syn
from oracle import gemm_nt, gemm_nt_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blackwell_programming_gb300 as gbmod
    gbmod.build()
    return gbmod


def make_ab(M, N, K, seed):
    """Seeded N(0,1) operands rounded to bf16 (the repository's generator)."""
    a = syn.f32_to_bf16_bits(syn.normals_f32(seed, 0, M * K)).reshape(M, K)
    b = syn.f32_to_bf16_bits(syn.normals_f32(seed, M * K, N * K)).reshape(N, K)
    return a, b


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def check_fp32(c_gpu, a64, b64, what):
    ref = gemm_nt(a64, b64)
    bound = a64.shape[1] * 2.0 ** -24 * (np.abs(a64) @ np.abs(b64).T)
    err = np.abs(c_gpu.astype(np.float64) - ref)
    worst = float(np.max(err - bound))
    assert worst <= 0.0, "%s: error exceeds the K-term sum bound by %.3e" % (what, worst)
    assert np.all(np.isfinite(c_gpu))


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64),      # one tile, one K step
    (300, 520, 136),     # ragged M, N and K
    (1, 2, 8),           # smallest legal problem
    (1000, 1000, 1000),  # several tiles in both directions, ragged everywhere
    (2048, 768, 4096),   # many K steps: the ring wraps many times
])
def test_gemm_parity(gb, M, N, K):
    a, b = make_ab(M, N, K, seed=M + N + K)
    da, db = to_dev(a), to_dev(b)
    gb.attn_check_device(reset=True)
    c32 = gb.gemm_nt(da, db, out_dtype=torch.float32)
    c16 = gb.gemm_nt(da, db)
    torch.cuda.synchronize()
    assert gb.attn_check_device(reset=True) == 0
    a64, b64 = syn.bf16_bits_to_f64(a), syn.bf16_bits_to_f64(b)
    check_fp32(c32.cpu().numpy(), a64, b64, "gemm %dx%dx%d" % (M, N, K))
    assert c16.dtype == torch.bfloat16 and torch.equal(c16, c32.to(torch.bfloat16))


def test_gemm_full_size_sampled_and_deterministic(gb):
    M, N, K = 16384, 6144, 4096   # the QKV projection of the GQA workload's model shape
    a, b = make_ab(M, N, K, seed=1)
    da, db = to_dev(a), to_dev(b)
    c1 = gb.gemm_nt(da, db, out_dtype=torch.float32)
    c2 = gb.gemm_nt(da, db, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    rows = [0, 1, 127, 128, 8191, 16255, 16383] + list(np.random.default_rng(2).integers(0, M, 9))
    a64, b64 = syn.bf16_bits_to_f64(a[rows]), syn.bf16_bits_to_f64(b)
    c = c1.cpu().numpy()[rows]
    ref = gemm_nt_rows(a64, b64, range(len(rows)))
    bound = K * 2.0 ** -24 * (np.abs(a64) @ np.abs(b64).T)
    assert float(np.max(np.abs(c - ref) - bound)) <= 0.0


@pytest.mark.parametrize("M,N,K", [(300, 520, 136), (2048, 768, 4096), (129, 256, 64), (256, 6, 8), (4096, 4096, 512)])
def test_pair_and_single_cta_kernels_agree(gb, M, N, K, monkeypatch):
    """M > 128 runs the CTA-pair kernel; ATTN_GEMM_SINGLE_CTA=1 forces the
    one-CTA kernel.  Both meet the bound; they sum each element's K products
    in the same 16-deep steps, so they agree to the last bit."""
    a, b = make_ab(M, N, K, seed=3 * M + N + K)
    da, db = to_dev(a), to_dev(b)
    gb.attn_check_device(reset=True)
    c_pair = gb.gemm_nt(da, db, out_dtype=torch.float32)
    monkeypatch.setenv("ATTN_GEMM_SINGLE_CTA", "1")
    c_single = gb.gemm_nt(da, db, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert gb.attn_check_device(reset=True) == 0
    a64, b64 = syn.bf16_bits_to_f64(a), syn.bf16_bits_to_f64(b)
    if M * N * K <= 2048 * 768 * 4096:
        check_fp32(c_pair.cpu().numpy(), a64, b64, "pair")
    else:
        rows = list(range(0, M, 97))
        ref = gemm_nt_rows(a64, b64, rows)
        bound = K * 2.0 ** -24 * (np.abs(a64[rows]) @ np.abs(b64).T)
        assert float(np.max(np.abs(c_pair.cpu().numpy()[rows] - ref) - bound)) <= 0.0
    assert torch.equal(c_pair, c_single)
