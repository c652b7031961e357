"""The Python binding's own checks, without a GPU: every refusal below is
raised while marshalling arguments, before any call reaches the library or
the CUDA runtime."""

import pytest

torch = pytest.importorskip("torch")

import deepseek_sparse_attention_row_gb300 as dsa  # noqa: E402


def test_logits_dtypes():
    assert dsa._logits_kind(torch.zeros(2)) == (torch.float32, "")
    assert dsa._logits_kind(torch.zeros(2, dtype=torch.bfloat16)) == (torch.bfloat16, "_bf16")
    with pytest.raises(TypeError, match="float32 or bfloat16"):
        dsa._logits_kind(torch.zeros(2, dtype=torch.float16))


def test_pointer_checks():
    assert dsa._dev_ptr(None, torch.int32, "row_ks", allow_none=True) is None
    with pytest.raises(ValueError, match="row_ke is required"):
        dsa._dev_ptr(None, torch.int32, "row_ke")
    with pytest.raises(TypeError, match="must be torch.int32"):
        dsa._dev_ptr(torch.zeros(3, dtype=torch.int64), torch.int32, "row_ke")
    # pageable host memory is never handed to a kernel
    with pytest.raises(ValueError, match="pinned host tensor"):
        dsa._dev_ptr(torch.zeros(3), torch.float32, "logits")
    with pytest.raises(ValueError, match="pinned host tensor"):
        dsa.mapped_host_pointer(torch.zeros(3))


def test_row_major_layout():
    x = torch.zeros(4, 6)
    assert dsa._row_major(x, "logits") == 6
    assert dsa._row_major(x[:, :5], "logits") == 6  # a column slice keeps the row stride
    with pytest.raises(ValueError, match="unit stride"):
        dsa._row_major(x.t(), "logits")


def test_host_calls_take_the_copy_path_for_pageable_inputs():
    # only pinned inputs are read in place; anything else is staged through the device
    assert not dsa._all_pinned(torch.zeros(2), None)
    assert dsa._all_pinned(None, None)

