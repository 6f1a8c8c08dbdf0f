"""GPU parity of token-major attention (attn_fwd_bshd) and of the layer slice
(attn_layer_fwd: QKV GEMM -> attention -> O GEMM) against the fp64 oracles.

Bars, each derived from the arithmetic of the step it checks:
* attn_fwd_bshd runs the prefill kernel of attn_fwd with other tensor-map
  coordinates and output strides, so on the same values its O and LSE equal
  attn_fwd's bit for bit; against the oracle the attention bar holds
  (max |dO| 2e-2, mean 2e-3, LSE 1e-3 relative).
* QKV: the oracle rounds the exact product to bf16, the GPU rounds an fp32
  sum of K exact products, so |dQKV| <= K 2^-24 (|X||W|^T) + one bf16 unit
  in the last place (2^-7 of the value's binade, at most 2^-7 |value|).
* O: the attention bar plus one bf16 unit of O (both sides round O).
* Y = O W_o^T, fp32 out: Y_gpu - Y_oracle = dO W_o^T + (fp32 sum error), so
  |dY| <= |dO| |W_o|^T + K 2^-24 |O_gpu| |W_o|^T elementwise, with dO the
  measured difference of the two O's (Hoelder's inequality, no slack).
"""
import numpy as np
import pytest

from blackwell_programming_gb300 import synthetic as syn
from oracle import attention, layer, layer_rows, round_bf16
from parity_util import LSE_REL, O_MAX_ABS, O_MEAN_ABS, check

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def token_major(buf, B, N, col0, H, d):
    """[B, N, H, d] view of columns [col0, col0 + H*d) of a [B*N, ld] buffer."""
    ld = buf.shape[1]
    return torch.as_strided(buf, (B, N, H, d), (N * ld, ld, d, 1), buf.storage_offset() + col0)


# ------------------------------------------------------------ attn_fwd_bshd

BSHD_CASES = [
    # B, Hq, Hkv, Nq, Nkv, d, causal
    (1, 2, 2, 128, 128, 64, False),
    (2, 4, 2, 200, 200, 128, True),        # ragged tail, GQA 2
    (1, 8, 2, 333, 333, 64, True),         # ragged, GQA 4
    (2, 4, 1, 100, 300, 128, True),        # Nq < Nkv: bottom-right causal alignment
    (1, 2, 1, 1, 77, 64, False),           # a single query
    (3, 4, 4, 513, 513, 128, False),       # several tiles plus a one-row tail
]


@pytest.mark.parametrize("case", BSHD_CASES, ids=lambda c: "B%d_H%d_%d_N%d_%d_d%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full"))
@pytest.mark.parametrize("o_fp32", [True, False], ids=["o32", "o16"])
def test_bshd_equals_head_major_and_oracle(gb, case, o_fp32):
    B, Hq, Hkv, Nq, Nkv, d, causal = case
    wl = syn.Workload("bshd", B, Hq, Hkv, Nq, Nkv, d, d, causal, 1.0 / np.sqrt(d), seed=sum(case))
    inp = syn.make_inputs(wl)
    q, k, v = (to_dev(t) for t in (inp.q, inp.k, inp.v))
    odt = torch.float32 if o_fp32 else torch.bfloat16
    o_ref_gpu, lse_ref_gpu = gb.attn_fwd(q, k, v, causal=causal, scale=wl.scale, out_dtype=odt)
    # Q in one padded token-major buffer, K and V side by side in another
    pad = 24
    qbuf = torch.full((B * Nq, Hq * d + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    kvbuf = torch.full((B * Nkv, 2 * Hkv * d + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    qt = token_major(qbuf, B, Nq, 0, Hq, d)
    kt = token_major(kvbuf, B, Nkv, 0, Hkv, d)
    vt = token_major(kvbuf, B, Nkv, Hkv * d, Hkv, d)
    qt.copy_(q.transpose(1, 2))
    kt.copy_(k.transpose(1, 2))
    vt.copy_(v.transpose(1, 2))
    # O into a padded buffer whose padding must stay untouched
    obuf = torch.full((B * Nq, Hq * d + pad), -3.0, dtype=odt, device="cuda")
    ot = token_major(obuf, B, Nq, 0, Hq, d)
    gb.attn_check_device(reset=True)
    _, lse = gb.attn_fwd_bshd(qt, kt, vt, causal=causal, scale=wl.scale, out=ot)
    status_ok(gb)
    assert torch.equal(ot.transpose(1, 2), o_ref_gpu), "O differs from the head-major call"
    assert torch.equal(lse, lse_ref_gpu), "LSE differs from the head-major call"
    assert bool((obuf[:, Hq * d:] == -3.0).all()), "padding of O was written"
    q64, k64, v64 = inp.f64()
    o_or, lse_or = attention(q64, k64, v64, causal, wl.scale)
    o_gpu = ot.transpose(1, 2).float().cpu().numpy()
    if o_fp32:
        check(o_gpu, lse.cpu().numpy(), o_or, lse_or, "bshd")
    else:
        d_o = np.abs(o_gpu - o_or) - 2.0 ** -8 * np.abs(o_or)
        assert float(d_o.max()) <= O_MAX_ABS and float(np.abs(o_gpu - o_or).mean()) <= O_MEAN_ABS + 2e-3


def test_bshd_rejects_bad_strides(gb):
    B, N, H, d = 1, 64, 2, 64
    buf = torch.zeros((B * N, H * d + 4), dtype=torch.bfloat16, device="cuda")   # ld % 8 != 0
    qt = token_major(buf, B, N, 0, H, d)
    with pytest.raises(ValueError):
        gb.attn_fwd_bshd(qt, qt, qt)
    # the C entry point itself refuses a token stride below the heads' width
    good = torch.zeros((B * N, H * d), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(good)
    import ctypes
    L = gb.load_library()
    st = L.attn_fwd_bshd(ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(o.data_ptr()), None,
                         B, H, H, N, N, d, H * d - 8, H * d, H * d, H * d, 0, 0, ctypes.c_float(0.1), None)
    assert st == gb.ATTN_ERR_INVALID_ARG
    st = L.attn_fwd_bshd(ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(good.data_ptr()),
                         ctypes.c_void_p(good.data_ptr()), ctypes.c_void_p(o.data_ptr()), None,
                         B, H, H, N, N, 96, H * d, H * d, H * d, H * d, 0, 0, ctypes.c_float(0.1), None)
    assert st == gb.ATTN_ERR_UNSUPPORTED


# ---------------------------------------------------------------- the layer

def check_qkv(qkv_gpu, x64, w64, qkv_or, what):
    bound = x64.shape[1] * 2.0 ** -24 * (np.abs(x64) @ np.abs(w64).T) + 2.0 ** -7 * np.abs(qkv_or)
    worst = float(np.max(np.abs(qkv_gpu - qkv_or) - bound))
    assert worst <= 0.0, "%s: QKV off by %.3e beyond its bound" % (what, worst)


def check_o(o_gpu, o_or, what):
    d = np.abs(o_gpu - o_or)
    assert float(np.max(d - 2.0 ** -7 * np.abs(o_or))) <= O_MAX_ABS, "%s: max |dO| %.3e" % (what, d.max())
    assert float(d.mean()) <= O_MEAN_ABS + 2.0 ** -8 * float(np.abs(o_or).mean()), \
        "%s: mean |dO| %.3e" % (what, d.mean())


def check_y(y_gpu, o_gpu, o_or, wo64, y_or, what, y_bf16=False):
    dO = np.abs(o_gpu - o_or)
    bound = dO @ np.abs(wo64).T + wo64.shape[1] * 2.0 ** -24 * (np.abs(o_gpu) @ np.abs(wo64).T)
    if y_bf16:
        bound = bound + 2.0 ** -7 * np.abs(y_or) + 2.0 ** -7 * bound
    worst = float(np.max(np.abs(y_gpu - y_or) - bound))
    assert worst <= 1e-12, "%s: Y off by %.3e beyond |dO||W_o|^T" % (what, worst)


LAYER_CASES = [
    # B, N, d_model, Hq, Hkv, d, causal
    (2, 300, 256, 4, 2, 64, True),
    (2, 300, 256, 4, 2, 64, False),
    (1, 520, 512, 4, 1, 128, True),
    (3, 129, 136, 2, 2, 128, True),       # d_model not a multiple of the GEMM's 64-deep step
]


@pytest.mark.parametrize("case", LAYER_CASES, ids=lambda c: "B%d_N%d_D%d_H%d_%d_d%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full"))
def test_layer_parity(gb, case):
    B, N, D, Hq, Hkv, d, causal = case
    lw = syn.LayerWorkload("layer", B, N, D, Hq, Hkv, d, causal, seed=sum(case))
    x, w_qkv, w_o = syn.make_layer_inputs(lw)
    dx, dwq, dwo = to_dev(x), to_dev(w_qkv), to_dev(w_o)
    gb.attn_check_device(reset=True)
    y, qkv, o, lse = gb.attn_layer_fwd(dx.view(B, N, D), dwq, dwo, Hq, Hkv, causal=causal, scale=lw.scale,
                                       y_dtype=torch.float32, want_lse=True)
    status_ok(gb)
    # each step agrees bit for bit with the library's own stand-alone calls
    assert torch.equal(qkv.view(B * N, -1), gb.gemm_nt(dx, dwq))
    assert torch.equal(y.view(B * N, -1), gb.gemm_nt(o.view(B * N, -1), dwo, out_dtype=torch.float32))
    # against the oracle
    x64, wq64, wo64 = (syn.bf16_bits_to_f64(t) for t in (x, w_qkv, w_o))
    y_or, qkv_or, o_or, lse_or = layer(x64, wq64, wo64, B, N, Hq, Hkv, causal, lw.scale)
    qkv_g = qkv.view(B * N, -1).double().cpu().numpy()
    o_g = o.view(B * N, -1).double().cpu().numpy()
    y_g = y.view(B * N, -1).double().cpu().numpy()
    check_qkv(qkv_g, x64, wq64, qkv_or, "layer")
    check_o(o_g, o_or, "layer")
    le = np.abs(lse.cpu().numpy() - lse_or) / np.maximum(1.0, np.abs(lse_or))
    assert float(le.max()) <= LSE_REL
    check_y(y_g, o_g, o_or, wo64, y_or, "layer")


def test_layer_full_size_sampled(gb):
    """The benchmarked layer (4 x 4096 tokens, d_model 4096, 32/8 heads of 128,
    causal, bf16 Y) in the bench's launch configuration; oracle rows of the
    last sequence."""
    lw = syn.LAYER_WORKLOADS["layer_gqa_d128"]
    B, N, D = lw.B, lw.N, lw.d_model
    x, w_qkv, w_o = syn.make_layer_inputs(lw)
    dx, dwq, dwo = to_dev(x), to_dev(w_qkv), to_dev(w_o)
    gb.attn_check_device(reset=True)
    y, qkv, o, _ = gb.attn_layer_fwd(dx.view(B, N, D), dwq, dwo, lw.Hq, lw.Hkv, causal=lw.causal, scale=lw.scale)
    status_ok(gb)
    assert bool(torch.isfinite(y).all())
    b = B - 1
    toks = [0, 1, 127, 128, 255, 2047, 3000, N - 1]
    rows = [b * N + t for t in toks]
    x64, wq64, wo64 = (syn.bf16_bits_to_f64(t) for t in (x, w_qkv, w_o))
    y_or, qkv_or, o_or = layer_rows(x64, wq64, wo64, B, N, lw.Hq, lw.Hkv, lw.causal, lw.scale, b, toks)
    qkv_g = qkv.view(B * N, -1)[rows].double().cpu().numpy()
    o_g = o.view(B * N, -1)[rows].double().cpu().numpy()
    y_g = y.view(B * N, -1)[rows].double().cpu().numpy()
    check_qkv(qkv_g, x64[rows], wq64, qkv_or, "full-size")
    check_o(o_g, o_or, "full-size")
    check_y(y_g, o_g, o_or, wo64, y_or, "full-size", y_bf16=True)
