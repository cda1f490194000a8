"""Host-side argument marshalling of the Python binding (no GPU): dtype, device, shape and
stride checks, and the narrowing of int64 sparse indices to the C ABI's int32 (ids beyond
int32 keep their meaning: negative stays masked, too large stays out of range)."""
import numpy as np
import pytest
import torch

import mla_latent_cache_attention_gb300 as m

CPU = torch.device("cpu")


def test_need_accepts_and_rejects():
    t = torch.zeros((4, 8), dtype=torch.int32)
    assert m._need(t, "x", (torch.int32,), CPU, ndim=2, contiguous=True) is t
    with pytest.raises(TypeError, match="dtype"):
        m._need(t, "x", (torch.int64,), CPU)
    with pytest.raises(ValueError, match="dimensions"):
        m._need(t, "x", (torch.int32,), CPU, ndim=1)
    with pytest.raises(ValueError, match="contiguous"):
        m._need(t.t(), "x", (torch.int32,), CPU, contiguous=True, inner=False)
    with pytest.raises(ValueError, match="innermost"):
        m._need(t.t(), "x", (torch.int32,), CPU)
    with pytest.raises(ValueError, match="expected"):
        m._need(t, "x", (torch.int32,), torch.device("cuda", 0))
    with pytest.raises(TypeError):
        m._need(np.zeros(3), "x", (torch.int32,), CPU)


def test_int32_indices_pass_through():
    idx = torch.tensor([0, 5, -1, 7], dtype=torch.int32)
    assert m._index_i32(idx, "kv_indices", CPU, -1, 100) is idx


def test_int64_indices_narrow_with_their_meaning():
    idx = torch.tensor([0, 5, -1, -(1 << 40), 99, (1 << 33) + 5, 2 ** 31], dtype=torch.int64)
    out = m._index_i32(idx, "kv_indices", CPU, -1, 100)
    assert out.dtype == torch.int32
    # valid ids unchanged; every negative id -> -1 (masked); every id >= 100 -> 100 (out of
    # range, masked and reported by the kernel) -- never wrapped onto a valid id
    assert out.tolist() == [0, 5, -1, -1, 99, 100, 100]


def test_int64_indptr_narrow():
    ptr = torch.tensor([0, 3, 3, 9], dtype=torch.int64)
    assert m._index_i32(ptr, "kv_indptr", CPU, 0, 9).tolist() == [0, 3, 3, 9]


def test_strided_or_2d_indices_are_rejected():
    idx = torch.arange(16, dtype=torch.int64)[::2]
    with pytest.raises(ValueError, match="contiguous"):
        m._index_i32(idx, "kv_indices", CPU, -1, 100)
    with pytest.raises(ValueError, match="dimensions"):
        m._index_i32(torch.zeros((2, 2), dtype=torch.int32), "kv_indices", CPU, -1, 100)
    with pytest.raises(TypeError, match="dtype"):
        m._index_i32(torch.zeros(4, dtype=torch.int16), "kv_indices", CPU, -1, 100)


def test_entry_points_reject_cpu_tensors():
    q = torch.zeros((1, 16, 576), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        m.sparse_fwd(q, torch.zeros((1, 656), dtype=torch.uint8), torch.zeros(2, dtype=torch.int32),
                     torch.zeros(1, dtype=torch.int32), 0.1)
    with pytest.raises(ValueError, match="CUDA"):
        m.paged_decode(q, torch.zeros((1, 64, 1152), dtype=torch.uint8), torch.zeros((1, 1), dtype=torch.int32),
                       torch.ones(1, dtype=torch.int32), fmt="bf16", max_context=64, softmax_scale=0.1)


def test_cache_geometry():
    c = torch.zeros((5, 64, 656), dtype=torch.uint8)
    assert m._cache_geometry(c) == (5, 64 * 656, 656, 64)
    assert m._cache_geometry(c.view(5, 1, 64, 656)) == (5, 64 * 656, 656, 64)
    with pytest.raises(ValueError, match="kv_cache"):
        m._cache_geometry(torch.zeros((5, 64), dtype=torch.uint8))
