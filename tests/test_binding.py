"""Binding checks that need no GPU: dtype, device, rank, shape and stride
validation happens in Python before any CUDA call (the binding pitfalls listed
in "Distilling a 4.5 hour CUDA talk", section 14)."""
import pytest
import torch

import blackwell_programming_gb300 as gb


@pytest.fixture(scope="module", autouse=True)
def built():
    gb.build()


def t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_rejects_wrong_dtype():
    with pytest.raises(TypeError):
        gb.attn_fwd(t(1, 1, 8, 64, dtype=torch.float16), t(1, 1, 8, 64), t(1, 1, 8, 64))


def test_rejects_cpu_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        gb.attn_fwd(t(1, 1, 8, 64), t(1, 1, 8, 64), t(1, 1, 8, 64))


def test_rejects_non_tensor():
    with pytest.raises(TypeError):
        gb.attn_fwd([1, 2], t(1, 1, 8, 64), t(1, 1, 8, 64))


def test_rejects_wrong_rank():
    with pytest.raises((TypeError, ValueError)):
        gb.attn_fwd(t(1, 8, 64), t(1, 1, 8, 64), t(1, 1, 8, 64))


def test_library_missing_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        gb.load_library(str(tmp_path / "nope.so"))
