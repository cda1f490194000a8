"""Pins of the oracle's chunked-context pieces ("vllm.models.kimi_k3.nvidia.mla":
_gather_context_latent and merge_attn_states in _forward_prefill_fused): the gather against an
independent walk of each request's pages and library casts of the dequantised values, and the
prefix / suffix merge against closed forms and the split invariance of attention."""
import numpy as np
import pytest
import torch

from mla_latent_cache_attention_gb300 import synth


def paged(seed, fmt, lens, bs=16):
    case = synth.paged_case(seed, fmt, B=len(lens), q_len=1, H=1, L_lo=1, L_hi=max(lens), block_size=bs,
                            seq_lens=lens)
    return case


def request_stream(case, b):
    """All entries of request b, in position order: the pages of its block-table row laid end
    to end (an independent walk of the paged layout)."""
    nblk = -(-int(case.seq_lens[b]) // case.cache.shape[1])
    pages = [case.cache[case.block_table[b, j]] for j in range(nblk)]
    return np.concatenate(pages, axis=0)[: case.seq_lens[b]]


def chunk(case, starts, lens):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cu, np.asarray(starts, dtype=np.int32)


@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP8, synth.DS_MLA])
def test_raw_gather_is_the_stored_entries(orc, fmt):
    case = paged(800 + fmt, fmt, [37, 100, 5, 64])
    starts, lens = [3, 50, 0, 16], [30, 50, 5, 48]
    cu, ss = chunk(case, starts, lens)
    got = orc.gather_context(fmt, case.cache, case.block_table, cu, ss, raw=True)
    eb = synth.ENTRY_BYTES[fmt]
    ref = np.concatenate([request_stream(case, b)[s:s + n, :eb] for b, (s, n) in enumerate(zip(starts, lens))])
    assert np.array_equal(got, ref)


def test_bf16_gather_equals_raw_and_no_starts_means_zero(orc):
    case = paged(810, synth.BF16, [20, 70])
    cu, _ = chunk(case, [0, 0], [20, 70])
    a = orc.gather_context(synth.BF16, case.cache, case.block_table, cu, None)
    b = orc.gather_context(synth.BF16, case.cache, case.block_table, cu, np.zeros(2, np.int32), raw=True)
    assert np.array_equal(a, b.view(np.uint16))


def test_fp8_upconvert_matches_library_casts(orc):
    case = paged(820, synth.FP8, [40, 33], bs=16)
    cu, ss = chunk(case, [5, 0], [35, 33])
    scale = 0.05
    got = orc.gather_context(synth.FP8, case.cache, case.block_table, cu, ss, scale=scale)
    raw = orc.gather_context(synth.FP8, case.cache, case.block_table, cu, ss, raw=True)
    f = torch.from_numpy(raw).view(torch.float8_e4m3fn).float() * torch.tensor(scale, dtype=torch.float32)
    assert np.array_equal(got, f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_ds_mla_upconvert_matches_library_casts(orc):
    case = paged(830, synth.DS_MLA, [50, 130], bs=64)
    cu, ss = chunk(case, [10, 1], [40, 129])
    got = orc.gather_context(synth.DS_MLA, case.cache, case.block_table, cu, ss)
    raw = orc.gather_context(synth.DS_MLA, case.cache, case.block_table, cu, ss, raw=True)
    codes = torch.from_numpy(raw[:, :512].copy()).view(torch.float8_e4m3fn).float()
    scales = torch.from_numpy(raw[:, 512:528].copy().view(np.float32))          # [n, 4]
    nope = (codes.view(-1, 4, 128) * scales[:, :, None]).view(-1, 512)            # fp32 products
    ref = torch.cat([nope.to(torch.bfloat16), torch.from_numpy(raw[:, 528:656].copy()).view(torch.bfloat16)], dim=1)
    assert np.array_equal(got, ref.view(torch.int16).numpy().view(np.uint16))


def test_rows_past_the_chunk_and_bad_blocks(orc):
    case = paged(840, synth.BF16, [10, 10])
    cu, ss = chunk(case, [0, 0], [10, 10])
    got = orc.gather_context(synth.BF16, case.cache, case.block_table, cu, ss, num_tokens=25)
    assert got.shape == (25, 576) and np.all(got[20:] == 0)
    bt = case.block_table.copy()
    bt[1, 0] = case.cache.shape[0] + 2
    with pytest.raises(ValueError):
        orc.gather_context(synth.BF16, case.cache, bt, cu, ss)


def bf(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_merge_closed_forms(orc):
    rng = np.random.default_rng(1)
    T, H, D = 3, 2, 128
    a, b = bf(rng.standard_normal((T, H, D))), bf(rng.standard_normal((T, H, D)))
    fa = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()
    fb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()
    lse = rng.standard_normal((H, T)).astype(np.float32) * 5
    out, l = orc.merge_attn_states(a, lse, b, lse)                      # equal weights: the mean
    np.testing.assert_allclose(out, (fa + fb) / 2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, lse.astype(np.float64) + np.log(2.0), rtol=0, atol=1e-12)
    ninf = np.full((H, T), -np.inf, dtype=np.float32)
    out, l = orc.merge_attn_states(a, lse, b, ninf)                     # an empty suffix
    assert np.array_equal(out, fa) and np.array_equal(l, lse.astype(np.float64))
    out, l = orc.merge_attn_states(a, ninf, b, ninf)                    # both empty
    assert np.all(out == 0) and np.all(l == -np.inf)
    gap = np.log(3.0)
    out, _ = orc.merge_attn_states(a, lse + np.float32(gap), b, lse)    # weights 3/4 and 1/4
    np.testing.assert_allclose(out, 0.75 * fa + 0.25 * fb, rtol=0, atol=1e-6)


def test_merge_is_attention_over_the_union(orc):
    c = synth.sparse_case(850, T=3, H=4, N=200, per_row=90, p_invalid=0.0, replace=False)
    cut = 40
    rows_a = [c.indices[c.indptr[t]:c.indptr[t] + cut] for t in range(3)]
    rows_b = [c.indices[c.indptr[t] + cut:c.indptr[t + 1]] for t in range(3)]

    def attend(rows):
        ptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
        return orc.sparse_fwd(c.q, c.records, ptr, np.concatenate(rows).astype(np.int32), c.softmax_scale, False)

    oa, la = attend(rows_a)
    ob, lb = attend(rows_b)
    full, lfull = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, False)
    out, l = orc.merge_attn_states(bf(oa), la.T.astype(np.float32), bf(ob), lb.T.astype(np.float32))
    # the partials enter as bf16 and their lse as fp32: within those roundings of the union
    assert np.all(np.abs(out - full) <= 2.0 ** -8 * (np.abs(oa) + np.abs(ob)) + 1e-12)
    np.testing.assert_allclose(l, lfull.T, rtol=0, atol=1e-5)
