"""Python binding of the C ABI in include/gbattn.h (ctypes, argument marshalling only).

Every entry point here has the name of the C function it calls.  Torch is used
for device memory and streams; all arithmetic runs in the library's kernels.
There is no fallback: if libgbattn.so is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_NO_DEVICE = 5
ATTN_ERR_SCRATCH_LIMIT = 6

# Symbols the shared library exports (the declarations of include/gbattn.h).
EXPORTS = ("attn_fwd", "attn_fwd_bf16out", "attn_check_device", "attn_status_string", "attn_last_cuda_error",
           "attn_version", "attn_decode_workspace_bytes", "attn_decode_fwd_noalloc", "gemm_bf16_nt",
           "attn_fwd_bshd", "attn_layer_fwd", "attn_fwd_dropout")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


def load_library(path: str | None = None):
    """Load libgbattn.so (built in-tree by ``_build.build``) and declare its ABI."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError("libgbattn.so is not built (expected at %s); call "
                           "blackwell_programming_gb300.build() first" % path)
    L = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
    L.attn_fwd.restype = i
    L.attn_fwd_bf16out.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
    L.attn_fwd_bf16out.restype = i
    ll = ctypes.c_longlong
    L.attn_fwd_bshd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, ll, ll, ll, ll, i, i, f, vp]
    L.attn_fwd_bshd.restype = i
    L.attn_layer_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    L.attn_layer_fwd.restype = i
    L.attn_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, f, ctypes.c_ulonglong, vp]
    L.attn_fwd_dropout.restype = i
    L.gemm_bf16_nt.argtypes = [vp, vp, vp, i, i, i, i, vp]
    L.gemm_bf16_nt.restype = i
    L.attn_check_device.argtypes = [vp, i]
    L.attn_check_device.restype = i
    L.attn_status_string.argtypes = [i]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_last_cuda_error.argtypes = []
    L.attn_last_cuda_error.restype = ctypes.c_char_p
    L.attn_version.argtypes = []
    L.attn_version.restype = i
    L.attn_decode_workspace_bytes.argtypes = [i, i, i]
    L.attn_decode_workspace_bytes.restype = ctypes.c_size_t
    L.attn_decode_fwd_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, f, vp]
    L.attn_decode_fwd_noalloc.restype = i
    if path == _build.LIB:
        _lib = L
    return L


def _raise(L, status: int, what: str):
    msg = "%s: %s" % (what, L.attn_status_string(status).decode())
    extra = L.attn_last_cuda_error().decode()
    if extra:
        msg += " (" + extra + ")"
    raise AttnError(status, msg)


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(status).decode()


def attn_last_cuda_error() -> str:
    return load_library().attn_last_cuda_error().decode()


def attn_version() -> int:
    return load_library().attn_version()


def attn_decode_workspace_bytes(B: int, Hkv: int, Nkv: int) -> int:
    return load_library().attn_decode_workspace_bytes(B, Hkv, Nkv)


# Size of the static scratch array behind attn_decode_fwd_noalloc (see gbattn.h).
NOALLOC_SCRATCH_BYTES = 48 << 20


def attn_decode_fwd_noalloc(q_ptr: int, kv_ptr: int, o_ptr: int, lse_ptr: int, B: int, Hq: int, Hkv: int,
                            Nkv: int, scale: float, stream_ptr: int = 0) -> int:
    """The allocation-free decode call with raw integer pointers; returns the status code.

    For callers that cannot let the library allocate device memory: the
    split partials go to the library's fixed static scratch array.
    """
    L = load_library()
    return L.attn_decode_fwd_noalloc(ctypes.c_void_p(q_ptr), ctypes.c_void_p(kv_ptr), ctypes.c_void_p(o_ptr),
                                     ctypes.c_void_p(lse_ptr), B, Hq, Hkv, Nkv, ctypes.c_float(scale),
                                     ctypes.c_void_p(stream_ptr))


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def attn_check_device(stream=None, reset: bool = False, device=None) -> int:
    """Synchronise the stream and read the kernels' error word (0 = ok)."""
    L = load_library()
    return L.attn_check_device(_stream_handle(stream, device), 1 if reset else 0)


def attn_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, Hq: int, Hkv: int,
                 Nq: int, Nkv: int, d_qk: int, d_v: int, causal: bool, scale: float, stream_ptr: int = 0) -> int:
    """The C call with raw integer pointers; returns the status code."""
    L = load_library()
    return L.attn_fwd(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                      ctypes.c_void_p(o_ptr), ctypes.c_void_p(lse_ptr), B, Hq, Hkv, Nq, Nkv, d_qk, d_v,
                      1 if causal else 0, ctypes.c_float(scale), ctypes.c_void_p(stream_ptr))


def attn_fwd_dropout(q, k, v, p_drop: float, seed: int, causal: bool = False, scale: float | None = None,
                     out=None, lse=None, want_lse: bool = True, stream=None):
    """Attention with dropout on the softmax weights (attn_fwd_dropout in gbattn.h).

    q: bf16 [B, Hq, Nq, d]; k, v: bf16 [B, Hkv, Nkv, d]; d 64 or 128, all
    contiguous.  p_drop = 0 or in [1/512, 1) (a nonzero p below 1/512 would
    round to no dropout and is refused); seed: 64-bit integer.  Returns (o fp32
    [B, Hq, Nq, d], lse fp32 [B, Hq, Nq] or None).
    """
    import torch
    L = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4:
            raise TypeError("%s must be a 4-D bfloat16 CUDA tensor [B, H, N, d]" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nkv, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    if out is None:
        out = torch.empty((B, Hq, Nq, d), dtype=torch.float32, device=dev)
    elif out.shape != (B, Hq, Nq, d) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 [B, Hq, Nq, d] tensor")
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = L.attn_fwd_dropout(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
                                B, Hq, Hkv, Nq, Nkv, d, d, 1 if causal else 0, ctypes.c_float(scale),
                                ctypes.c_float(p_drop), ctypes.c_ulonglong(seed & 0xFFFFFFFFFFFFFFFF),
                                _stream_handle(stream, dev))
    if st != ATTN_OK:
        _raise(L, st, "attn_fwd_dropout")
    return out, lse


def gemm_raw(a_ptr: int, b_ptr: int, c_ptr: int, M: int, N: int, K: int, c_fp32: bool,
             stream_ptr: int = 0) -> int:
    """The C call gemm_bf16_nt with raw integer pointers; returns the status code."""
    L = load_library()
    return L.gemm_bf16_nt(ctypes.c_void_p(a_ptr), ctypes.c_void_p(b_ptr), ctypes.c_void_p(c_ptr), M, N, K,
                          1 if c_fp32 else 0, ctypes.c_void_p(stream_ptr))


def gemm_nt(a, b, out=None, out_dtype=None, stream=None):
    """C = A B^T on the GPU: a bf16 [M, K], b bf16 [N, K] (a linear layer's
    weight), both contiguous on one CUDA device; C [M, N] bf16 (default) or
    fp32.  Work is queued on ``stream`` (default: the current stream)."""
    import torch
    L = load_library()
    for name, t in (("a", a), ("b", b)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 2:
            raise TypeError("%s must be a 2-D bfloat16 CUDA tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if a.device != b.device:
        raise ValueError("a and b must be on one device")
    M, K = a.shape
    N, Kb = b.shape
    if Kb != K:
        raise ValueError("shape mismatch: a %s b %s" % (tuple(a.shape), tuple(b.shape)))
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("C is fp32 or bf16, not %s" % out_dtype)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    elif out.shape != (M, N) or out.dtype != out_dtype or not out.is_contiguous() or out.device != a.device:
        raise ValueError("out must be a contiguous %s [M, N] tensor on a's device" % out_dtype)
    with torch.cuda.device(a.device):
        st = L.gemm_bf16_nt(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                            ctypes.c_void_p(out.data_ptr()), M, N, K, 1 if out_dtype == torch.float32 else 0,
                            _stream_handle(stream, a.device))
    if st != ATTN_OK:
        _raise(L, st, "gemm_bf16_nt")
    return out


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             want_lse: bool = True, stream=None, out_dtype=None):
    """O = softmax(mask(scale * Q K^T)) V and LSE on the GPU.

    q: bf16 [B, Hq, Nq, d_qk]; k: bf16 [B, Hkv, Nkv, d_qk];
    v: bf16 [B, Hkv, Nkv, d_v], or the view ``k[..., :d_v]`` of k (the latent
    layout where V is the first d_v features of K).  All on one CUDA device,
    contiguous (a view of k is accepted for v as described).  scale defaults
    to 1/sqrt(d_qk).  Returns (o [B, Hq, Nq, d_v], lse fp32 [B, Hq, Nq] or
    None).  O is fp32 (attn_fwd), or bf16 when ``out_dtype`` is
    torch.bfloat16 or ``out`` is a bf16 tensor (attn_fwd_bf16out).  Work is
    queued on ``stream`` (default: the current stream).
    """
    import torch
    L = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % name)
        if t.dtype != torch.bfloat16:
            raise TypeError("%s must be bfloat16, got %s" % (name, t.dtype))
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if t.dim() != 4:
            raise ValueError("%s must be 4-D [B, H, N, d]" % name)
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    B, Hq, Nq, d_qk = q.shape
    Bk, Hkv, Nkv, dk = k.shape
    Bv, Hv, Nv, d_v = v.shape
    if Bk != B or Bv != B or Hv != Hkv or Nv != Nkv or dk != d_qk:
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if not q.is_contiguous() or not k.is_contiguous():
        raise ValueError("q and k must be contiguous [B, H, N, d] row-major tensors")
    aliased = (v.data_ptr() == k.data_ptr() and d_v < d_qk and v.stride() == k.stride())
    if not aliased and not v.is_contiguous():
        raise ValueError("v must be contiguous, or the view k[..., :d_v]")
    if scale is None:
        scale = 1.0 / math.sqrt(d_qk)
    dev = q.device
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.float32
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("O is fp32 or bf16, not %s" % out_dtype)
    if out is None:
        out = torch.empty((B, Hq, Nq, d_v), dtype=out_dtype, device=dev)
    elif out.shape != (B, Hq, Nq, d_v) or out.dtype != out_dtype or not out.is_contiguous() or out.device != dev:
        raise ValueError("out must be a contiguous %s [B, Hq, Nq, d_v] tensor on q's device" % out_dtype)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    elif lse is not None and (lse.shape != (B, Hq, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Nq] tensor")
    v_ptr = k.data_ptr() if aliased else v.data_ptr()
    fn = L.attn_fwd if out_dtype == torch.float32 else L.attn_fwd_bf16out
    with torch.cuda.device(dev):
        st = fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v_ptr),
                        ctypes.c_void_p(out.data_ptr()),
                        ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
                        B, Hq, Hkv, Nq, Nkv, d_qk, d_v, 1 if causal else 0, ctypes.c_float(scale),
                        _stream_handle(stream, dev))
    if st != ATTN_OK:
        _raise(L, st, fn.__name__)
    return out, lse


def _token_major_ld(name, t, heads, d):
    """Token stride (elements) of a [B, N, H, d] tensor whose heads sit side by
    side in each token's row, as attn_fwd_bshd reads it."""
    B, N, H, dd = t.shape
    if H != heads or dd != d:
        raise ValueError("%s must be [B, N, %d, %d], got %s" % (name, heads, d, tuple(t.shape)))
    sb, sn, sh, sc = t.stride()
    if sc != 1 or sh != d or sn % 8 != 0 or sn < heads * d or (B > 1 and sb != N * sn):
        raise ValueError("%s must be token-major: strides (N*ld, ld, d, 1) with ld %% 8 == 0 and "
                         "ld >= H*d, got %s" % (name, t.stride()))
    if t.data_ptr() % 16 != 0:
        raise ValueError("%s must start on a 16-byte boundary" % name)
    return sn


def attn_fwd_bshd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                  want_lse: bool = True, stream=None, out_dtype=None):
    """Attention on token-major tensors (attn_fwd_bshd in gbattn.h).

    q: bf16 [B, Nq, Hq, d], k and v: bf16 [B, Nkv, Hkv, d], d 64 or 128, each
    with strides (N * ld, ld, d, 1): for example column slices of a QKV
    projection's output viewed as [B, N, H, d].  Returns (o [B, Nq, Hq, d],
    lse fp32 [B, Hq, Nq] or None); O is bf16 unless ``out_dtype`` (or
    ``out``) says fp32.
    """
    import torch
    L = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4:
            raise TypeError("%s must be a 4-D bfloat16 CUDA tensor [B, N, H, d]" % name)
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    B, Nq, Hq, d = q.shape
    Bk, Nkv, Hkv, _ = k.shape
    if Bk != B or v.shape[0] != B or v.shape[1] != Nkv:
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    q_ld = _token_major_ld("q", q, Hq, d)
    k_ld = _token_major_ld("k", k, Hkv, d)
    v_ld = _token_major_ld("v", v, Hkv, d)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("O is fp32 or bf16, not %s" % out_dtype)
    if out is None:
        out = torch.empty((B, Nq, Hq, d), dtype=out_dtype, device=dev)
    elif out.dtype != out_dtype or out.device != dev or out.dim() != 4 or out.shape[:2] != (B, Nq):
        raise ValueError("out must be a %s [B, Nq, Hq, d] tensor on q's device" % out_dtype)
    o_ld = _token_major_ld("out", out, Hq, d)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    elif lse is not None and (lse.shape != (B, Hq, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Nq] tensor")
    with torch.cuda.device(dev):
        st = L.attn_fwd_bshd(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                             ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                             ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
                             B, Hq, Hkv, Nq, Nkv, d, q_ld, k_ld, v_ld, o_ld,
                             1 if out_dtype == torch.float32 else 0, 1 if causal else 0, ctypes.c_float(scale),
                             _stream_handle(stream, dev))
    if st != ATTN_OK:
        _raise(L, st, "attn_fwd_bshd")
    return out, lse


def attn_layer_raw(x_ptr: int, w_qkv_ptr: int, w_o_ptr: int, qkv_ptr: int, o_ptr: int, y_ptr: int, lse_ptr: int,
                   B: int, N: int, d_model: int, Hq: int, Hkv: int, d: int, causal: bool, scale: float,
                   y_fp32: bool, stream_ptr: int = 0) -> int:
    """The C call attn_layer_fwd with raw integer pointers; returns the status code."""
    L = load_library()
    return L.attn_layer_fwd(*(ctypes.c_void_p(p) for p in (x_ptr, w_qkv_ptr, w_o_ptr, qkv_ptr, o_ptr, y_ptr,
                                                          lse_ptr)),
                            B, N, d_model, Hq, Hkv, d, 1 if causal else 0, ctypes.c_float(scale),
                            1 if y_fp32 else 0, ctypes.c_void_p(stream_ptr))


def attn_layer_fwd(x, w_qkv, w_o, Hq: int, Hkv: int, causal: bool = True, scale: float | None = None,
                   y_dtype=None, want_lse: bool = False, qkv=None, o=None, y=None, stream=None):
    """Y = Attn(X W_qkv^T) W_o^T (attn_layer_fwd in gblayer.h).

    x: bf16 [B, N, d_model]; w_qkv: bf16 [(Hq + 2 Hkv) d, d_model] (W_q rows,
    then W_k, then W_v); w_o: bf16 [d_model, Hq d].  Returns (y [B, N,
    d_model], qkv bf16 [B, N, (Hq + 2 Hkv) d], o bf16 [B, N, Hq d], lse fp32
    [B, Hq, N] or None); y is bf16 unless ``y_dtype`` is torch.float32.
    """
    import torch
    L = load_library()
    for name, t, nd in (("x", x, 3), ("w_qkv", w_qkv, 2), ("w_o", w_o, 2)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != nd:
            raise TypeError("%s must be a %d-D bfloat16 CUDA tensor" % (name, nd))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    B, N, d_model = x.shape
    rows, kq = w_qkv.shape
    if kq != d_model or rows % (Hq + 2 * Hkv) != 0:
        raise ValueError("w_qkv must be [(Hq + 2 Hkv) d, d_model], got %s" % (tuple(w_qkv.shape),))
    d = rows // (Hq + 2 * Hkv)
    if tuple(w_o.shape) != (d_model, Hq * d):
        raise ValueError("w_o must be [d_model, Hq d] = %s, got %s" % ((d_model, Hq * d), tuple(w_o.shape)))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if y_dtype is None:
        y_dtype = y.dtype if y is not None else torch.bfloat16
    dev = x.device

    def buf(t, shape, dtype, name):
        if t is None:
            return torch.empty(shape, dtype=dtype, device=dev)
        if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous() or t.device != dev:
            raise ValueError("%s must be a contiguous %s %s tensor on x's device" % (name, dtype, shape))
        return t

    qkv = buf(qkv, (B, N, rows), torch.bfloat16, "qkv")
    o = buf(o, (B, N, Hq * d), torch.bfloat16, "o")
    y = buf(y, (B, N, d_model), y_dtype, "y")
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev) if want_lse else None
    with torch.cuda.device(dev):
        st = L.attn_layer_fwd(*(ctypes.c_void_p(t.data_ptr()) for t in (x, w_qkv, w_o, qkv, o, y)),
                              ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
                              B, N, d_model, Hq, Hkv, d, 1 if causal else 0, ctypes.c_float(scale),
                              1 if y_dtype == torch.float32 else 0, _stream_handle(stream, dev))
    if st != ATTN_OK:
        _raise(L, st, "attn_layer_fwd")
    return y, qkv, o, lse
