"""Pins of the oracle's sparse forward with the general op's extras (attention sink, second key
segment; "vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla", flydsl_sparse_mla_fp8ds_supported
argument list): reductions to the pinned plain sparse forward, the sink's closed forms, and
the union of two segments."""
import numpy as np

from mla_latent_cache_attention_gb300 import synth


def case(seed=0, T=5, H=4, N=120, per_row=40, p_invalid=0.1):
    return synth.sparse_case(seed, T=T, H=H, N=N, per_row=per_row, p_invalid=p_invalid, replace=True, ragged=True)


def test_no_extras_is_the_plain_forward(orc):
    c = case(1)
    a = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    b = orc.sparse_fwd_ext(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    ninf = np.full(c.q.shape[1], -np.inf, dtype=np.float32)
    d = orc.sparse_fwd_ext(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True, attn_sink=ninf)
    assert np.array_equal(a[0], d[0]) and np.array_equal(a[1], d[1])


def test_sink_closed_forms(orc):
    c = case(2)
    H = c.q.shape[1]
    o, l = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    sink = np.linspace(-3, 40, H).astype(np.float32)
    os_, ls = orc.sparse_fwd_ext(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True, attn_sink=sink)
    s64 = sink.astype(np.float64)[None, :]
    fin = np.isfinite(l)
    ref_l = np.where(fin, np.logaddexp(l, s64), s64)               # empty row: lse = sink
    np.testing.assert_allclose(ls, ref_l, rtol=0, atol=1e-12)
    scale = np.where(fin, np.exp(l - ls), 0.0)                       # out shrinks by e^{lse - lse_sink}
    np.testing.assert_allclose(os_, o * scale[:, :, None], rtol=1e-12, atol=1e-13)


def test_single_key_with_equal_sink_halves_the_value(orc):
    c = case(3, T=1, H=2, N=10, per_row=1, p_invalid=0.0)
    c.indptr = np.array([0, 1], dtype=np.int32)
    c.indices = np.array([4], dtype=np.int32)
    o, l = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, False)
    os_, ls = orc.sparse_fwd_ext(c.q, c.records, c.indptr, c.indices, c.softmax_scale, False,
                                 attn_sink=l[0].astype(np.float32))
    v = orc.decode_entry(synth.DS_MLA, c.records[4])[:512]
    np.testing.assert_allclose(os_[0], 0.5 * np.broadcast_to(v, (2, 512)), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(ls[0], l[0] + np.log(2.0), rtol=0, atol=1e-6)


def test_second_segment_is_the_union(orc):
    c = case(4, T=4, H=3, N=150, per_row=60)
    rng = np.random.default_rng(4)
    extra = synth.ds_mla_records(rng, 70)
    n2 = rng.integers(0, 30, size=4)
    ip2 = np.concatenate([[0], np.cumsum(n2)]).astype(np.int32)
    ix2 = rng.integers(0, 70, size=ip2[-1]).astype(np.int32)
    ix2[rng.random(ix2.size) < 0.1] = -1
    o, l = orc.sparse_fwd_ext(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True, extra_records=extra,
                              extra_indptr=ip2, extra_indices=ix2)
    # the same keys as one list over one pool holding both record sets
    pool = np.concatenate([c.records, extra])
    rows = [np.concatenate([c.indices[c.indptr[t]:c.indptr[t + 1]],
                            np.where(ix2[ip2[t]:ip2[t + 1]] >= 0, ix2[ip2[t]:ip2[t + 1]] + 150, -1)]) for t in range(4)]
    ptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    ro, rl = orc.sparse_fwd(c.q, pool, ptr, np.concatenate(rows).astype(np.int32), c.softmax_scale, True)
    np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


def test_empty_row_with_sink(orc):
    c = synth.config0()                          # row 3 is empty
    sink = np.full(c.q.shape[1], 2.5, dtype=np.float32)
    o, l = orc.sparse_fwd_ext(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True, attn_sink=sink)
    assert np.all(o[3] == 0) and np.all(l[3] == 2.5)
