"""Fused attention forward for one NVIDIA GB300 (sm_103a).

The compute path is libgbattn.so (hand-written CUDA with tcgen05, TMA and
mbarrier inline PTX) behind the C ABI of include/gbattn.h (attention) and
include/gbgemm.h and include/gblayer.h (the projection GEMMs around it and
the layer slice they form); this package is a thin
ctypes binding over it plus the seeded synthetic-input generator.
"""
from . import _build
from .binding import (ATTN_ERR_CUDA, ATTN_ERR_INVALID_ARG, ATTN_ERR_NO_DEVICE, ATTN_ERR_SCRATCH_LIMIT,
                      ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED, ATTN_OK, EXPORTS, AttnError,
                      attn_check_device, attn_decode_fwd_noalloc,
                      attn_decode_workspace_bytes, attn_fwd, attn_fwd_raw, attn_last_cuda_error,
                      attn_status_string,
                      attn_version, attn_fwd_bshd, attn_fwd_dropout, attn_layer_fwd, attn_layer_raw, gemm_nt, gemm_raw,
                      load_library)


def build(force: bool = False) -> str:
    """Compile libgbattn.so for sm_103a (if stale) and load it."""
    path = _build.build(force=force)
    load_library()
    return path


__all__ = ["build", "attn_fwd", "attn_fwd_raw", "attn_check_device", "attn_status_string",
           "attn_version", "attn_decode_workspace_bytes", "attn_last_cuda_error", "AttnError", "load_library", "EXPORTS",
           "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_CUDA",
           "ATTN_ERR_TIMEOUT", "ATTN_ERR_NO_DEVICE", "ATTN_ERR_SCRATCH_LIMIT", "attn_decode_fwd_noalloc",
           "gemm_nt", "gemm_raw", "attn_fwd_bshd", "attn_layer_fwd", "attn_layer_raw", "attn_fwd_dropout"]
