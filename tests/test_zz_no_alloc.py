"""The allocation-free decode entry point, attn_decode_fwd_noalloc.

Some callers cannot let a library allocate device memory while they run (a
framework whose caching allocator already holds the GPU's free memory, a
serving loop with a fixed memory budget, a plug-in whose host forbids
allocation).  For them the library's split-KV decode has a variant whose
partial results live in a fixed static device array instead of a
stream-ordered pool workspace.  These checks call it through the C ABI and hold
its output to the same tolerance as every other parity test, against the fp64
oracle and against the regular attn_fwd path on two calls in a row (the array
keeps the previous call's contents, so the second call must not depend on it
being clear).

The file is named to be collected last, so a failure here leaves every other
test already run.
"""
import math

import numpy as np
import pytest

from blackwell_programming_gb300 import synthetic as syn
from tests.parity_util import LSE_REL, O_MAX_ABS, O_MEAN_ABS, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blackwell_programming_gb300 as gbmod
    gbmod.build()
    return gbmod


def _close(o_a, l_a, o_b, l_b):
    d = (o_a.double() - o_b.double()).abs()
    assert float(d.max()) <= O_MAX_ABS
    assert float(d.mean()) <= O_MEAN_ABS
    rel = (l_a.double() - l_b.double()).abs() / torch.clamp(l_b.double().abs(), min=1.0)
    assert float(rel.max()) <= LSE_REL


@pytest.mark.parametrize("B,Hq,Hkv,Nkv", [(8, 128, 1, 2000), (3, 64, 2, 1111)])
def test_noalloc_matches_attn_fwd_twice(gb, B, Hq, Hkv, Nkv):
    wl = syn.Workload("noalloc", B, Hq, Hkv, 1, Nkv, 576, 512, False, 1 / math.sqrt(192), v_aliases_k=True)
    inp = syn.make_inputs(wl)
    q, k, v = to_torch(inp)
    stream = torch.cuda.current_stream().cuda_stream
    o_ref, l_ref = gb.attn_fwd(q, k, v, causal=False, scale=wl.scale)
    torch.cuda.synchronize()
    for call in range(2):
        o = torch.full((B, Hq, 1, 512), float("nan"), device="cuda")
        lse = torch.full((B, Hq, 1), float("nan"), device="cuda")
        st = gb.attn_decode_fwd_noalloc(q.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        B, Hq, Hkv, Nkv, wl.scale, stream)
        assert st == gb.ATTN_OK, (call, gb.attn_status_string(st), gb.attn_last_cuda_error())
        torch.cuda.synchronize()
        assert gb.attn_check_device(reset=True) == 0
        assert torch.isfinite(o).all() and torch.isfinite(lse).all(), call
        _close(o, lse, o_ref, l_ref)


def test_noalloc_matches_the_oracle(gb):
    """attn_decode_fwd_noalloc against the fp64 oracle directly, element by
    element, on a case whose rows merge several split pieces."""
    from oracle import attention
    wl = syn.Workload("noalloc_oracle", 2, 32, 1, 1, 700, 576, 512, False, 1 / math.sqrt(192), v_aliases_k=True)
    inp = syn.make_inputs(wl)
    q, k, _ = to_torch(inp)
    o = torch.full((wl.B, wl.Hq, 1, 512), float("nan"), device="cuda")
    lse = torch.full((wl.B, wl.Hq, 1), float("nan"), device="cuda")
    st = gb.attn_decode_fwd_noalloc(q.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr(), wl.B, wl.Hq, wl.Hkv,
                                    wl.Nkv, wl.scale, torch.cuda.current_stream().cuda_stream)
    assert st == gb.ATTN_OK, (gb.attn_status_string(st), gb.attn_last_cuda_error())
    torch.cuda.synchronize()
    assert gb.attn_check_device(reset=True) == 0
    qf, kf, vf = inp.f64()
    o_ref, lse_ref = attention(qf, kf, vf, False, wl.scale)
    d = np.abs(o.cpu().numpy() - o_ref)
    assert float(d.max()) <= O_MAX_ABS and float(d.mean()) <= O_MEAN_ABS
    rel = np.abs(lse.cpu().numpy() - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    assert float(rel.max()) <= LSE_REL


def test_noalloc_rejects_problems_beyond_the_static_scratch(gb):
    # 1024 sequences of 32 keys: every CTA's range crosses many (sequence,
    # half) segments, so the partials need more than the 48 MiB array.
    B, Hq, Hkv, Nkv = 1024, 128, 1, 32
    q = torch.zeros((B, Hq, 1, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((B, Hkv, Nkv, 576), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((B, Hq, 1, 512), device="cuda")
    st = gb.attn_decode_fwd_noalloc(q.data_ptr(), kv.data_ptr(), o.data_ptr(), 0, B, Hq, Hkv, Nkv, 0.07,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == gb.ATTN_ERR_SCRATCH_LIMIT
    assert "static array" in gb.attn_last_cuda_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0


def test_noalloc_reserves_no_device_memory(gb):
    # The property the entry point exists for: once the library is loaded on
    # the device (the first call), further calls take no device memory.  All
    # buffers are made before the measurement, so the only thing that could
    # move the device's free memory is the library itself.
    B, Hq, Hkv, Nkv = 16, 128, 1, 4096
    wl = syn.Workload("noalloc_mem", B, Hq, Hkv, 1, Nkv, 576, 512, False, 1 / math.sqrt(192), v_aliases_k=True)
    q, k, _ = to_torch(syn.make_inputs(wl))
    o = torch.empty((B, Hq, 1, 512), device="cuda")
    lse = torch.empty((B, Hq, 1), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        st = gb.attn_decode_fwd_noalloc(q.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        B, Hq, Hkv, Nkv, wl.scale, stream)
        assert st == gb.ATTN_OK, (gb.attn_status_string(st), gb.attn_last_cuda_error())

    call()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert gb.attn_check_device(reset=True) == 0
