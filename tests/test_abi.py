"""The C-ABI library builds, loads and exports what include/*.h declare.

These run without a GPU: only calls that return before touching CUDA are made
(argument checks), no compute.
"""
import ctypes
import os
import re

import pytest

import blackwell_programming_gb300 as gb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    gb.build()
    return gb.load_library()


def declared_functions():
    """Every function the headers in include/ declare."""
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:attn|gemm)_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_abi():
    assert declared_functions() == sorted(gb.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exported_symbols_via_nm(lib):
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", gb._build.LIB], capture_output=True, text=True).stdout
    names = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in names, name


def test_version_and_strings(lib):
    assert gb.attn_version() == 100
    assert gb.attn_status_string(gb.ATTN_OK) == "ok"
    assert gb.attn_status_string(gb.ATTN_ERR_INVALID_ARG) == "invalid argument"
    assert gb.attn_status_string(gb.ATTN_ERR_TIMEOUT) == "kernel wait timed out"
    assert gb.attn_status_string(12345) == "unknown status"


GOOD = dict(B=1, Hq=2, Hkv=1, Nq=128, Nkv=128, d_qk=128, d_v=128, causal=False, scale=0.1)
P = 1 << 20   # a 16-byte-aligned fake address; never dereferenced because the checks fail first


def call(**kw):
    a = dict(GOOD)
    ptrs = dict(q_ptr=P, k_ptr=P * 2, v_ptr=P * 3, o_ptr=P * 4, lse_ptr=P * 5)
    for key in list(kw):
        if key in ptrs:
            ptrs[key] = kw.pop(key)
    a.update(kw)
    return gb.attn_fwd_raw(ptrs["q_ptr"], ptrs["k_ptr"], ptrs["v_ptr"], ptrs["o_ptr"], ptrs["lse_ptr"],
                           a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nkv"], a["d_qk"], a["d_v"], a["causal"],
                           a["scale"])


@pytest.mark.parametrize("bad", [
    dict(q_ptr=0), dict(k_ptr=0), dict(v_ptr=0), dict(o_ptr=0),
    dict(B=0), dict(Hq=0), dict(Hkv=-1), dict(Nq=0), dict(Nkv=0), dict(d_qk=0), dict(d_v=0),
    dict(Hq=3, Hkv=2),
    dict(scale=float("nan")), dict(scale=float("inf")), dict(scale=-1.0),
    dict(q_ptr=P + 8), dict(k_ptr=P + 2), dict(o_ptr=P + 4), dict(lse_ptr=P + 2),
])
def test_invalid_arguments_rejected_before_any_cuda_call(lib, bad):
    assert call(**bad) == gb.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [
    dict(d_qk=96, d_v=96), dict(d_qk=128, d_v=64), dict(d_qk=256, d_v=256),
    dict(d_qk=576, d_v=512, Nq=2),                        # latent prefill needs v == k
    dict(d_qk=576, d_v=512, Nq=1),                        # latent decode needs v == k
    dict(d_qk=576, d_v=512, Nq=64, causal=1, v_ptr=P * 3),   # a separate V is not the latent layout
])
def test_unsupported_shapes(lib, bad):
    assert call(**bad) == gb.ATTN_ERR_UNSUPPORTED


def test_v_longer_than_k_alias_rejected(lib):
    assert call(v_ptr=P * 2, d_qk=64, d_v=128) == gb.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [
    dict(a=0), dict(b=0), dict(c=0), dict(M=0), dict(N=-2), dict(K=0),
    dict(K=12),          # rows of A and B must be whole 16-byte units
    dict(N=7),           # C columns are stored in pairs
    dict(a=P + 8), dict(b=P + 4), dict(c=P + 2),
])
def test_gemm_invalid_arguments(lib, bad):
    a = dict(a=P, b=P * 2, c=P * 3, M=256, N=512, K=128)
    a.update(bad)
    assert gb.gemm_raw(a["a"], a["b"], a["c"], a["M"], a["N"], a["K"], False) == gb.ATTN_ERR_INVALID_ARG


def test_gemm_sizes_past_32_bit_rows(lib):
    assert gb.gemm_raw(P, P * 2, P * 3, 1 << 20, 4096, 4096, False) == gb.ATTN_ERR_UNSUPPORTED


def _dropout_raw(lib, p_drop, d_qk=128, d_v=128, v_ptr=P * 3):
    import ctypes
    return lib.attn_fwd_dropout(ctypes.c_void_p(P), ctypes.c_void_p(P * 2), ctypes.c_void_p(v_ptr),
                                ctypes.c_void_p(P * 4), ctypes.c_void_p(P * 5), 1, 2, 1, 128, 128, d_qk, d_v, 0,
                                ctypes.c_float(0.1), ctypes.c_float(p_drop), ctypes.c_ulonglong(7), None)


@pytest.mark.parametrize("p_drop", [1.0, -0.1, float("nan"), 0.999, 2.0, 1e-3, 1.0 / 1024, 1e-30])
def test_dropout_probability_checked(lib, p_drop):
    # 0.999 is below 1 but rounds to t = 256, which would drop every weight;
    # a nonzero p below 1/512 rounds to t = 0 and would silently drop nothing
    assert _dropout_raw(lib, p_drop) == gb.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("p_drop", [0.0, 1.0 / 512, 0.1, 0.99])
def test_dropout_probability_accepted(lib, p_drop):
    # past the argument checks (without a GPU the call then fails on the device)
    assert _dropout_raw(lib, p_drop) != gb.ATTN_ERR_INVALID_ARG


def test_dropout_latent_shape_unsupported(lib):
    assert _dropout_raw(lib, 0.1, d_qk=576, d_v=512, v_ptr=P * 2) == gb.ATTN_ERR_UNSUPPORTED


def _bshd_raw(lib, q=P, d=128, H=2, q_ld=256, k_ld=256, v_ld=256, o_ld=256):
    import ctypes
    return lib.attn_fwd_bshd(ctypes.c_void_p(q), ctypes.c_void_p(P * 2), ctypes.c_void_p(P * 3),
                             ctypes.c_void_p(P * 4), None, 1, H, H, 64, 64, d, q_ld, k_ld, v_ld, o_ld, 0, 1,
                             ctypes.c_float(0.1), None)


@pytest.mark.parametrize("bad", [dict(q_ld=252), dict(k_ld=260), dict(o_ld=128), dict(v_ld=0), dict(q=P + 8)])
def test_bshd_invalid_arguments(lib, bad):
    assert _bshd_raw(lib, **bad) == gb.ATTN_ERR_INVALID_ARG


def test_bshd_unsupported_head_dim(lib):
    assert _bshd_raw(lib, d=96, q_ld=192, k_ld=192, v_ld=192, o_ld=192) == gb.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("bad,want", [
    (dict(x=0), gb.ATTN_ERR_INVALID_ARG), (dict(y=0), gb.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3), gb.ATTN_ERR_INVALID_ARG), (dict(N=0), gb.ATTN_ERR_INVALID_ARG),
    (dict(d=96), gb.ATTN_ERR_UNSUPPORTED),
])
def test_layer_invalid_arguments(lib, bad, want):
    a = dict(x=P, w_qkv=P * 2, w_o=P * 3, qkv=P * 4, o=P * 5, y=P * 6, B=1, N=64, d_model=256, Hq=4, Hkv=2, d=64)
    a.update(bad)
    assert gb.attn_layer_raw(a["x"], a["w_qkv"], a["w_o"], a["qkv"], a["o"], a["y"], 0, a["B"], a["N"],
                             a["d_model"], a["Hq"], a["Hkv"], a["d"], True, 0.1, False) == want
