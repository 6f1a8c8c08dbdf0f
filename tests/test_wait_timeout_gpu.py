"""Failure detection on the GPU without a fault: a bounded wait that runs out.

A test-only kernel (tests/cuda/wait_timeout.cu) uses the library's mbarrier
wait on barriers nothing ever arrives on.  The first wait must give up after
the library's limit (2 s), record block, warp, barrier and parity in the
error word and raise the CTA's abort flag; a second wait, started later,
must return through the abort flag instead of running its own limit; and
the CUDA context must stay usable (a normal attention call afterwards still
matches the oracle).
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
    out = str(tmp_path_factory.mktemp("wt") / "libwait_timeout.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-o", out, os.path.join(HERE, "cuda", "wait_timeout.cu")], check=True)
    L = ctypes.CDLL(out)
    L.run_wait_timeout.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    L.run_wait_timeout.restype = ctypes.c_int
    return L


def test_bounded_wait_gives_up_and_reports(lib):
    torch.cuda.init()
    err = np.zeros(8, dtype=np.uint32)
    exit_ns = np.zeros(2, dtype=np.uint64)
    res = np.zeros(4, dtype=np.uint32)
    assert lib.run_wait_timeout(err.ctypes.data, exit_ns.ctypes.data, res.ctypes.data) == 0
    assert err[0] == 1                      # timeout bit
    assert err[1] == 0 and err[2] == 0      # block 0, warp 0 gave up first
    assert err[3] == res[2]                 # on barrier 0's shared-memory address
    assert err[4] == 0                      # waiting for parity 0
    assert res[0] == 0 and res[1] == 0      # both waits report failure
    t0, t1 = exit_ns / 1e9
    assert 1.9 < t0 < 4.0                   # the limit is 2 s
    assert t1 < t0 + 0.5                    # warp 1 left through the abort flag, not its own limit


def test_context_still_usable_after_timeout(lib):
    import blackwell_programming_gb300 as gb
    from blackwell_programming_gb300 import synthetic as syn
    from oracle import attention
    from tests.parity_util import check, run_gpu
    gb.build()
    wl = syn.Workload("after_timeout", 1, 2, 1, 200, 200, 128, 128, True, 0.09)
    inp = syn.make_inputs(wl)
    o, lse = run_gpu(inp)
    q, k, v = inp.f64()
    o_ref, lse_ref = attention(q, k, v, True, 0.09)
    check(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "after timeout")
