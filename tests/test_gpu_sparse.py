"""GPU parity of the sparse forward (CSR over fp8_ds_mla records) against the fp64 oracle:
the tiny configuration in full, edge cases (empty / all-masked / ragged rows, duplicates,
head counts that are not multiples of 16, strided out, no lse, int64 indices), and the
full-size prefill configuration (T=4096, H=16, top-2048 of 65536 records) on all 4096 rows.

Every case runs both kernel designs of the library: mla_sparse_fwd (gather warps, codes
straight into the tensor cores) and the test aid mla_sparse_fwd_staged (bulk copies and an
exact e4m3 -> f16 conversion in shared memory)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import assert_attn_close, assert_lse_close, t_bf16, t_i32, t_i64, t_u8

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


@pytest.fixture(params=["gather", "staged"])
def kern(request):
    return request.param


_ORACLE_CACHE = {}


def oracle_sparse(c: synth.SparseCase, rows=None, key=None):
    """The oracle's result for a case (memoised by `key` for the full-size case, which both
    kernel designs compare against)."""
    if key is not None and key in _ORACLE_CACHE:
        return _ORACLE_CACHE[key]
    r = oracle.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, c.has_invalid, rows=rows)
    if key is not None:
        _ORACLE_CACHE[key] = r
    return r


def run(m, c: synth.SparseCase, rows=None, out=None, lse=True, kern="gather", key=None):
    q = t_bf16(c.q)
    o, l = m.sparse_fwd(q, t_u8(c.records), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=c.has_invalid, out=out, return_lse=lse, kernel=kern)
    ro, rl = oracle_sparse(c, rows=rows, key=key)
    if rows is not None:
        o = o[torch.as_tensor(rows, device=o.device)]
        l = l[torch.as_tensor(rows, device=o.device)] if l is not None else None
    return o, l, ro, rl


def test_config0_tiny(m, kern):
    c = synth.config0()
    o, l, ro, rl = run(m, c, kern=kern)
    assert_attn_close(o, ro, "config0 out")
    assert_lse_close(l, rl, "config0 lse")
    assert torch.all(o[3] == 0) and torch.all(l[3] == -np.inf)
    assert m.read_device_errors() == 0


def test_golden_warmup_problem(m, kern):
    g = json.load(open(os.path.join(GOLDEN, "warmup_one_token.json")))
    rec = torch.zeros((1, 656), dtype=torch.uint8, device="cuda")
    for H in g["heads"]:
        q = torch.zeros((1, H, 576), dtype=torch.bfloat16, device="cuda")
        o, l = m.sparse_fwd(q, rec, t_i32(g["indptr"]), t_i32(g["indices"]), g["softmax_scale"], return_lse=True,
                            kernel=kern)
        assert torch.all(o == g["expected_out"]) and torch.all(l == g["expected_lse"])


@pytest.mark.parametrize("H", [1, 5, 16, 20, 64, 96, 128])
def test_head_counts(m, kern, H):
    c = synth.sparse_case(100 + H, T=6, H=H, N=500, per_row=200, p_invalid=0.1, replace=True, ragged=True)
    o, l, ro, rl = run(m, c, kern=kern)
    assert_attn_close(o, ro, f"H={H}")
    assert_lse_close(l, rl, f"H={H}")


def test_multi_tile_ragged_rows(m, kern):
    # row lengths 0, 1, 127, 128, 129, 255, 256, 257, 1000, all-masked
    lens = [0, 1, 127, 128, 129, 255, 256, 257, 1000, 40]
    rng = np.random.default_rng(5)
    c = synth.sparse_case(5, T=len(lens), H=16, N=3000, per_row=1, p_invalid=0.0, replace=True)
    ptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = rng.integers(0, 3000, size=ptr[-1]).astype(np.int32)
    idx[rng.random(idx.size) < 0.07] = -1
    idx[ptr[-2]:ptr[-1]] = -1                    # last row fully masked
    c.q = synth.normal_bf16_bits(rng, (len(lens), 16, 576))
    c.indptr, c.indices, c.has_invalid = ptr, idx, True
    o, l, ro, rl = run(m, c, kern=kern)
    assert_attn_close(o, ro, "ragged")
    assert_lse_close(l, rl, "ragged")
    assert torch.all(o[0] == 0) and torch.all(o[-1] == 0)


def test_duplicates_without_has_invalid_and_no_lse(m, kern):
    c = synth.sparse_case(9, T=8, H=16, N=50, per_row=300, p_invalid=0.0, replace=True)
    o, l, ro, rl = run(m, c, lse=False, kern=kern)
    assert l is None
    assert_attn_close(o, ro, "duplicates")


def test_strided_out_and_q(m, kern):
    c = synth.sparse_case(13, T=5, H=16, N=400, per_row=150, p_invalid=0.05, replace=False)
    qbig = torch.zeros((5, 16, 640), dtype=torch.bfloat16, device="cuda")
    qbig[:, :, :576] = t_bf16(c.q)
    out = torch.full((5, 16, 600), 7.0, dtype=torch.bfloat16, device="cuda")
    o, l = m.sparse_fwd(qbig[:, :, :576], t_u8(c.records), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=True, out=out[:, :, :512], return_lse=True, kernel=kern)
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    assert_attn_close(out[:, :, :512], ro, "strided")
    assert torch.all(out[:, :, 512:] == 7.0)
    assert_lse_close(l, rl, "strided")


def test_padded_record_pitch(m, kern):
    c = synth.sparse_case(17, T=4, H=16, N=300, per_row=200, p_invalid=0.1, replace=True)
    padded = np.zeros((300, 672), dtype=np.uint8)
    padded[:, :656] = c.records
    o, l = m.sparse_fwd(t_bf16(c.q), t_u8(padded), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=True, return_lse=True, kernel=kern)
    ro, rl = oracle.sparse_fwd(c.q, padded, c.indptr, c.indices, c.softmax_scale, True)
    assert_attn_close(o, ro, "padded pitch")
    assert_lse_close(l, rl, "padded pitch")


def test_power_of_two_and_large_scales(m, kern):
    rng = np.random.default_rng(21)
    c = synth.sparse_case(21, T=4, H=16, N=256, per_row=256, p_invalid=0.0, replace=False)
    c.records[:, 512:528] = (2.0 ** rng.integers(-6, 8, size=(256, 4))).astype(np.float32).view(np.uint8)
    o, l, ro, rl = run(m, c, kern=kern)
    assert_attn_close(o, ro, "pow2 scales")
    # scales up to 2^7 put |lse| near 3e4, where fp32 resolution is 2e-3: allow 1e-6 relative
    assert_lse_close(l, rl, "pow2 scales", rel=1e-6)


def test_out_of_range_index_is_masked_and_flagged(m, kern):
    c = synth.sparse_case(23, T=3, H=16, N=100, per_row=50, p_invalid=0.0, replace=True)
    m.read_device_errors()
    bad = c.indices.copy()
    bad[7] = 100
    q = t_bf16(c.q)
    o, l = m.sparse_fwd(q, t_u8(c.records), t_i32(c.indptr), t_i32(bad), c.softmax_scale, return_lse=True,
                        kernel=kern)
    assert m.read_device_errors() & 1
    masked = bad.copy()
    masked[7] = -1
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, masked, c.softmax_scale, True)
    assert_attn_close(o, ro, "masked bad index")


def test_int64_indices_match_int32(m, kern):
    # the sparse forward's interface takes int32 or int64 kv_indptr / kv_indices; int64 ids
    # beyond int32 keep their meaning (negative: masked, too large: out of range)
    c = synth.sparse_case(29, T=5, H=16, N=300, per_row=140, p_invalid=0.1, replace=True, ragged=True)
    q, rec = t_bf16(c.q), t_u8(c.records)
    o32, l32 = m.sparse_fwd(q, rec, t_i32(c.indptr), t_i32(c.indices), c.softmax_scale, has_invalid=True,
                            return_lse=True, kernel=kern)
    i64 = c.indices.astype(np.int64)
    i64[i64 < 0] = -(1 << 40)
    o64, l64 = m.sparse_fwd(q, rec, t_i64(c.indptr), t_i64(i64), c.softmax_scale, has_invalid=True,
                            return_lse=True, kernel=kern)
    assert torch.equal(o32, o64) and torch.equal(l32, l64)
    assert m.read_device_errors() == 0
    big = c.indices.astype(np.int64)
    big[3] = (1 << 33) + 5                     # wraps to 5 if narrowed without a clamp
    o, l = m.sparse_fwd(q, rec, t_i64(c.indptr), t_i64(big), c.softmax_scale, has_invalid=True,
                        return_lse=True, kernel=kern)
    assert m.read_device_errors() & 1
    masked = c.indices.copy()
    masked[3] = -1
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, masked, c.softmax_scale, True)
    assert_attn_close(o, ro, "int64 out-of-range id")
    assert_lse_close(l, rl, "int64 out-of-range id")


def test_strided_indices_are_rejected(m):
    c = synth.sparse_case(31, T=2, H=16, N=100, per_row=20, p_invalid=0.0, replace=True)
    idx = t_i32(np.repeat(c.indices, 2))[::2]
    assert not idx.is_contiguous()
    with pytest.raises(ValueError, match="contiguous"):
        m.sparse_fwd(t_bf16(c.q), t_u8(c.records), t_i32(c.indptr), idx, c.softmax_scale)


@pytest.mark.slow
def test_config2_full_size_all_rows(m, kern):
    """Sparse prefill at full size (T=4096, H=16, 2048 indices per row over 65536 records,
    ~5 % masked): all 4096 rows x 16 heads compared with the oracle."""
    c = synth.config2()
    o, l, ro, rl = run(m, c, kern=kern, key="config2")
    assert_attn_close(o, ro, "config2")
    assert_lse_close(l, rl, "config2")
    assert m.read_device_errors() == 0


def test_row_chunks_on_two_concurrent_streams(m):
    """Row chunks alternating between two compute streams (so that consecutive chunk kernels
    overlap on the device, as a pipelined caller runs them) give the full call's result bit
    for bit; sampled rows also match the oracle."""
    c = synth.sparse_case(41, T=400, H=16, N=20000, per_row=1024, p_invalid=0.05, replace=False)
    q, rec, ptr, idx = t_bf16(c.q), t_u8(c.records), t_i32(c.indptr), t_i32(c.indices)
    o_full, l_full = m.sparse_fwd(q, rec, ptr, idx, c.softmax_scale, has_invalid=True, return_lse=True)
    out = torch.full_like(o_full, 3.0)
    lse = torch.full_like(l_full, 5.0)
    cur = torch.cuda.current_stream()
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    for st in streams:
        st.wait_stream(cur)
    bounds = [0, 40, 120, 200, 280, 360, 400]
    for i in range(len(bounds) - 1):
        r0, r1 = bounds[i], bounds[i + 1]
        with torch.cuda.stream(streams[i % 2]):
            m.sparse_fwd(q[r0:r1], rec, ptr[r0:r1 + 1], idx, c.softmax_scale, has_invalid=True,
                         out=out[r0:r1], return_lse=True, lse=lse[r0:r1])
    for st in streams:
        cur.wait_stream(st)
    torch.cuda.synchronize()
    assert torch.equal(out, o_full) and torch.equal(lse, l_full)
    rows = np.random.default_rng(41).choice(400, 8, replace=False)
    sub_ptr = np.concatenate([[0], np.cumsum([c.indptr[r + 1] - c.indptr[r] for r in rows])]).astype(np.int32)
    sub_idx = np.concatenate([c.indices[c.indptr[r]:c.indptr[r + 1]] for r in rows]).astype(np.int32)
    ro, rl = oracle.sparse_fwd(c.q[rows], c.records, sub_ptr, sub_idx, c.softmax_scale, True)
    sel = torch.as_tensor(rows, device=out.device)
    assert_attn_close(out[sel], ro, "two-stream chunks")
    assert_lse_close(lse[sel], rl, "two-stream chunks")


def test_row_chunks_through_indptr_slices(m, kern):
    """Rows served in chunks, each call given a slice of kv_indptr (first offset non-zero)
    over the whole kv_indices and slices of out / lse, give the full call's result bit for
    bit; chunks run on a second stream."""
    c = synth.sparse_case(37, T=11, H=16, N=900, per_row=300, p_invalid=0.1, replace=True, ragged=True)
    q, rec, ptr, idx = t_bf16(c.q), t_u8(c.records), t_i32(c.indptr), t_i32(c.indices)
    o_full, l_full = m.sparse_fwd(q, rec, ptr, idx, c.softmax_scale, has_invalid=True, return_lse=True, kernel=kern)
    out = torch.full_like(o_full, 3.0)
    lse = torch.full_like(l_full, 5.0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for r0, r1 in [(0, 3), (3, 4), (4, 10), (10, 11)]:
            m.sparse_fwd(q[r0:r1], rec, ptr[r0:r1 + 1], idx, c.softmax_scale, has_invalid=True,
                         out=out[r0:r1], return_lse=True, lse=lse[r0:r1], kernel=kern)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert torch.equal(out, o_full) and torch.equal(lse, l_full)
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    assert_attn_close(out, ro, "row chunks")
    assert_lse_close(lse, rl, "row chunks")
