"""GPU parity of the sparse forward's extras (mla_sparse_fwd_ext: attention sink, second key
segment, kv_splits) against the fp64 oracle, on ragged rows (empty, one key, tile edges, long),
with masked entries, and at the prefill configuration's density (2048 of 65536 records per
row) with every extra at once."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import assert_attn_close, assert_lse_close, t_bf16, t_i32, t_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def ragged_case(seed, H=16, N=3000, lens=(0, 1, 127, 128, 129, 300, 1000, 2048, 40)):
    rng = np.random.default_rng(seed)
    c = synth.sparse_case(seed, T=len(lens), H=H, N=N, per_row=1, p_invalid=0.0, replace=True)
    c.indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    c.indices = rng.integers(0, N, size=c.indptr[-1]).astype(np.int32)
    c.indices[rng.random(c.indices.size) < 0.07] = -1
    c.q = synth.normal_bf16_bits(rng, (len(lens), H, 576))
    c.has_invalid = True
    return c


def second_segment(seed, T, N2=500, hi=400):
    rng = np.random.default_rng(seed)
    rec = synth.ds_mla_records(rng, N2)
    n = rng.integers(0, hi, size=T)
    n[0] = 0
    ptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    idx = rng.integers(0, N2, size=ptr[-1]).astype(np.int32)
    idx[rng.random(idx.size) < 0.05] = -1
    return rec, ptr, idx


def run(m, c, *, sink=None, seg=None, kv_splits=1):
    kw = {}
    if seg is not None:
        kw = dict(extra_kv=t_u8(seg[0]), extra_indptr=t_i32(seg[1]), extra_indices=t_i32(seg[2]))
    o, l = m.sparse_fwd(t_bf16(c.q), t_u8(c.records), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=True, return_lse=True, kv_splits=kv_splits,
                        attn_sink=None if sink is None else torch.from_numpy(sink).cuda(), **kw)
    okw = {} if seg is None else dict(extra_records=seg[0], extra_indptr=seg[1], extra_indices=seg[2])
    ro, rl = oracle.sparse_fwd_ext(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True, attn_sink=sink, **okw)
    return o, l, ro, rl


@pytest.mark.parametrize("kv_splits", [2, 3, 8])
def test_kv_splits(m, kv_splits):
    c = ragged_case(60 + kv_splits)
    o, l, ro, rl = run(m, c, kv_splits=kv_splits)
    assert_attn_close(o, ro, f"kv_splits={kv_splits}")
    assert_lse_close(l, rl, f"kv_splits={kv_splits}")
    assert torch.all(o[0] == 0) and torch.all(l[0] == -np.inf)
    assert m.read_device_errors() == 0


def test_attn_sink(m):
    c = ragged_case(70, H=20)
    sink = np.linspace(-5.0, 25.0, 20).astype(np.float32)
    sink[3] = -np.inf                                              # a head without a sink
    o, l, ro, rl = run(m, c, sink=sink)
    assert_attn_close(o, ro, "sink")
    assert_lse_close(l, rl, "sink")
    assert torch.all(o[0] == 0)
    lg = l[0].cpu().numpy()                                        # the empty row: lse = sink
    assert np.array_equal(lg[np.isfinite(sink)], sink[np.isfinite(sink)]) and lg[3] == -np.inf


@pytest.mark.parametrize("kv_splits", [1, 3])
def test_second_segment(m, kv_splits):
    c = ragged_case(80 + kv_splits)
    seg = second_segment(81 + kv_splits, c.q.shape[0])
    o, l, ro, rl = run(m, c, seg=seg, kv_splits=kv_splits)
    assert_attn_close(o, ro, "second segment")
    assert_lse_close(l, rl, "second segment")


def test_everything_at_prefill_density(m):
    # 256 rows of the sparse-prefill configuration (2048 of 65536 records, ~5 % masked), a
    # second segment of up to 512 keys per row, a sink per head and 4 splits
    c = synth.config2(T=256)
    seg = second_segment(90, 256, N2=4096, hi=512)
    sink = np.random.default_rng(91).uniform(0, 30, 16).astype(np.float32)
    o, l, ro, rl = run(m, c, sink=sink, seg=seg, kv_splits=4)
    assert_attn_close(o, ro, "all extras")
    assert_lse_close(l, rl, "all extras")
    assert m.read_device_errors() == 0


def test_splits_agree_with_the_plain_kernel(m):
    c = synth.config2(T=64)
    q, rec, ptr, idx = t_bf16(c.q), t_u8(c.records), t_i32(c.indptr), t_i32(c.indices)
    o1, l1 = m.sparse_fwd(q, rec, ptr, idx, c.softmax_scale, has_invalid=True, return_lse=True)
    o4, l4 = m.sparse_fwd(q, rec, ptr, idx, c.softmax_scale, has_invalid=True, return_lse=True, kv_splits=4)
    assert torch.allclose(l1, l4, atol=1e-4, rtol=0)
    assert torch.allclose(o1.float(), o4.float(), atol=1e-2, rtol=1e-2)
