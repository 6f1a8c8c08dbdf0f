"""Shared helpers for the GPU parity tests: feed identical bf16 inputs to the
CUDA path and to the fp64 oracle, compare within the stated tolerances."""
from __future__ import annotations

import numpy as np

# Tolerances for fp32 O and LSE against the fp64 oracle (bf16 inputs, fp32
# accumulation, bf16 P inside the kernel).
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def to_torch(inp, device="cuda"):
    """bf16 device tensors from an Inputs record; V may be the view k[..., :d_v]."""
    import torch
    q = torch.from_numpy(inp.q.view(np.int16)).view(torch.bfloat16).to(device)
    k = torch.from_numpy(inp.k.view(np.int16)).view(torch.bfloat16).to(device)
    if inp.v is None:
        v = k[..., : inp.wl.d_v]
    else:
        v = torch.from_numpy(inp.v.view(np.int16)).view(torch.bfloat16).to(device)
    return q, k, v


def run_gpu(inp, stream=None):
    import torch
    import blackwell_programming_gb300 as gb
    wl = inp.wl
    q, k, v = to_torch(inp)
    gb.attn_check_device(reset=True)
    o, lse = gb.attn_fwd(q, k, v, causal=wl.causal, scale=wl.scale, stream=stream)
    torch.cuda.synchronize()
    st = gb.attn_check_device(reset=True)
    assert st == 0, "device status %d (%s): %s" % (st, gb.attn_status_string(st), gb.attn_last_cuda_error())
    return o, lse


def check(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Assert the parity bar and return (max |dO|, mean |dO|, max LSE err)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, what
    assert np.all(np.isfinite(o_gpu)), what + ": non-finite O"
    d = np.abs(o_gpu - o_ref)
    mx, mean = float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0
    # LSE: -inf exactly where the oracle has no visible key
    inf_ref = np.isinf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), inf_ref), what + ": -inf LSE pattern differs"
    fin = ~inf_ref
    le = np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    lmax = float(le.max()) if le.size else 0.0
    assert mx <= O_MAX_ABS, "%s: max |dO| %.3e" % (what, mx)
    assert mean <= O_MEAN_ABS, "%s: mean |dO| %.3e" % (what, mean)
    assert lmax <= LSE_REL, "%s: LSE error %.3e" % (what, lmax)
    return mx, mean, lmax
