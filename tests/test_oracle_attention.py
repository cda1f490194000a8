"""Pins of the oracle's attention (sparse forward, paged decode / spec-verify, LSE merge)
against closed forms, invariants and cross-API identities.  Decoding in these tests goes
through torch's CPU float8 / bfloat16 casts, never through the oracle."""
import json
import math
import os

import numpy as np
import pytest
import torch

from mla_latent_cache_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x) -> np.ndarray:
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def e4m3_codes(x) -> np.ndarray:
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def make_record(nope_vals, scales, rope_vals) -> np.ndarray:
    """A 656-byte record whose NoPE codes are e4m3(nope_vals) (exactly representable values)."""
    rec = np.zeros(656, dtype=np.uint8)
    rec[:512] = e4m3_codes(np.broadcast_to(nope_vals, (512,)))
    rec[512:528] = np.asarray(scales, dtype=np.float32).view(np.uint8)
    rec[528:656] = bf16_bits(np.broadcast_to(rope_vals, (64,))).view(np.uint8)
    return rec


def decoded_ds(rec: np.ndarray) -> np.ndarray:
    """Independent decode of ds_mla records [N, 656] -> [N, 576] f64 via torch casts."""
    rec = np.ascontiguousarray(rec)
    e = torch.from_numpy(rec[:, :512].copy()).view(torch.float8_e4m3fn).double().numpy()
    s = rec[:, 512:528].copy().view(np.float32).astype(np.float64)
    r = torch.from_numpy(rec[:, 528:656].copy().view(np.int16)).view(torch.bfloat16).double().numpy()
    return np.concatenate([e * np.repeat(s, 128, axis=1), r], axis=1)


def q_with(rope0: float, H: int = 1, T: int = 1) -> np.ndarray:
    q = np.zeros((T, H, 576), dtype=np.float32)
    q[:, :, 512] = rope0
    return bf16_bits(q)


# ---------------------------------------------------------------- golden: warmup problem

def test_golden_warmup_one_token(orc):
    g = json.load(open(os.path.join(GOLDEN, "warmup_one_token.json")))
    rec = np.zeros((1, 656), dtype=np.uint8)
    for H in g["heads"]:
        q = np.zeros((1, H, 576), dtype=np.uint16)
        out, lse = orc.sparse_fwd(q, rec, g["indptr"], g["indices"], g["softmax_scale"], False)
        assert np.all(out == g["expected_out"]) and np.all(lse == g["expected_lse"])


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_its_latent_and_logit(orc):
    rec = make_record(np.linspace(-4, 4, 512).round(0), [0.5, 2.0, 0.25, 1.5], 1.0)
    q = q_with(2.0)
    out, lse = orc.sparse_fwd(q, rec[None], [0, 1], [0], 0.125, False)
    assert np.array_equal(out[0, 0], decoded_ds(rec[None])[0, :512])
    assert lse[0, 0] == 2.0 * 1.0 * 0.125


def test_two_keys_with_log3_gap(orc):
    # x1 = ln3 * 1 * 1, x2 = 0  ->  weights 3/4 and 1/4, lse = ln 4
    r1 = make_record(1.0, [1, 1, 1, 1], 1.0)
    r2 = make_record(3.0, [1, 1, 1, 1], 0.0)
    recs = np.stack([r1, r2])
    out, lse = orc.sparse_fwd(q_with(1.0), recs, [0, 2], [0, 1], math.log(3.0), False)
    np.testing.assert_allclose(out[0, 0], np.full(512, 0.75 * 1 + 0.25 * 3), rtol=0, atol=1e-14)
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-14


def test_identical_keys_add_log_n(orc):
    rec = make_record(2.0, [0.5, 0.5, 0.5, 0.5], 3.0)
    for n in (1, 2, 7, 33):
        out, lse = orc.sparse_fwd(q_with(1.0), rec[None], [0, n], [0] * n, 0.5, False)
        np.testing.assert_allclose(out[0, 0], np.full(512, 1.0), atol=1e-13)
        assert abs(lse[0, 0] - (1.5 + math.log(n))) < 1e-13


def test_zero_scale_gives_mean_and_log_n(orc):
    c = synth.sparse_case(11, T=2, H=3, N=40, per_row=17, p_invalid=0.0, replace=True)
    out, lse = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, 0.0, False)
    V = decoded_ds(c.records)[:, :512]
    for t in range(2):
        idx = c.indices[c.indptr[t]:c.indptr[t + 1]]
        np.testing.assert_allclose(out[t], np.broadcast_to(V[idx].mean(0), (3, 512)), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[t], math.log(idx.size), atol=1e-13)


def test_large_scale_selects_argmax_key(orc):
    # rope[0] values 0..4 on five keys, q rope0 = 1 -> logits 0..4 * sigma; sigma huge -> key 4
    recs = np.stack([make_record(float(i + 1), [1, 1, 1, 1], float(i)) for i in range(5)])
    out, lse = orc.sparse_fwd(q_with(1.0), recs, [0, 5], [2, 4, 0, 3, 1], 1e4, False)
    np.testing.assert_allclose(out[0, 0], np.full(512, 5.0), rtol=1e-12)
    assert abs(lse[0, 0] - 4e4) < 1e-9


def test_constant_values_sum_of_weights_is_one(orc):
    rng = np.random.default_rng(3)
    recs = np.stack([make_record(2.0, [0.25, 0.25, 0.25, 0.25], float(rng.integers(-5, 5))) for _ in range(20)])
    q = q_with(1.3, H=2)
    out, lse = orc.sparse_fwd(q, recs, [0, 20], np.arange(20), 0.9, False)
    np.testing.assert_allclose(out[0], 0.5, rtol=1e-13)
    # independent log-sum-exp of the logits
    x = 0.9 * float(torch.tensor(1.3).to(torch.bfloat16)) * decoded_ds(recs)[:, 512]
    assert abs(lse[0, 0] - float(torch.logsumexp(torch.tensor(x), 0))) < 1e-12


# ---------------------------------------------------------------- masking / empty rows

def test_masked_and_empty_rows(orc):
    c = synth.config0()
    out, lse = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    assert np.all(out[3] == 0) and np.all(np.isneginf(lse[3]))
    # a row made only of -1 entries is empty as well
    out2, lse2 = orc.sparse_fwd(c.q[:1], c.records, [0, 3], [-1, -1, -1], c.softmax_scale, True)
    assert np.all(out2 == 0) and np.all(np.isneginf(lse2))


def test_negative_index_without_has_invalid_is_an_error(orc):
    c = synth.config0()
    with pytest.raises(ValueError):
        orc.sparse_fwd(c.q[:1], c.records, [0, 2], [0, -1], 0.1, False)
    with pytest.raises(ValueError):
        orc.sparse_fwd(c.q[:1], c.records, [0, 1], [256], 0.1, True)


def test_permutation_and_padding_invariance(orc):
    c = synth.sparse_case(21, T=3, H=4, N=64, per_row=29, p_invalid=0.2, replace=True)
    out, lse = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    rng = np.random.default_rng(0)
    idx2, ptr2 = [], [0]
    for t in range(3):
        row = c.indices[c.indptr[t]:c.indptr[t + 1]].copy()
        rng.shuffle(row)
        row = np.concatenate([row, [-1] * (t + 2)])
        rng.shuffle(row)
        idx2.extend(row)
        ptr2.append(len(idx2))
    out2, lse2 = orc.sparse_fwd(c.q, c.records, ptr2, idx2, c.softmax_scale, True)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-13)


def test_duplicate_key_counts_twice(orc):
    c = synth.sparse_case(5, T=1, H=2, N=16, per_row=5, p_invalid=0.0, replace=False)
    out, lse = orc.sparse_fwd(c.q, c.records, [0, 1], c.indices[:1], 0.3, False)
    out2, lse2 = orc.sparse_fwd(c.q, c.records, [0, 2], np.repeat(c.indices[:1], 2), 0.3, False)
    np.testing.assert_allclose(out2, out, rtol=1e-13)
    np.testing.assert_allclose(lse2, lse + math.log(2), atol=1e-13)


def test_row_selection_matches_full(orc):
    c = synth.sparse_case(8, T=6, H=3, N=50, per_row=10, p_invalid=0.1, replace=True)
    out, lse = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, 0.2, True)
    o2, l2 = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, 0.2, True, rows=[5, 0, 3])
    assert np.array_equal(o2, out[[5, 0, 3]]) and np.array_equal(l2, lse[[5, 0, 3]])


# ---------------------------------------------------------------- merge (split invariance)

def test_merge_of_split_results_equals_unsplit(orc):
    c = synth.sparse_case(13, T=1, H=2, N=80, per_row=60, p_invalid=0.0, replace=False)
    out, lse = orc.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, False)
    cuts = [0, 7, 8, 31, 60]
    parts, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = orc.sparse_fwd(c.q, c.records, [0, b - a], c.indices[a:b], c.softmax_scale, False)
        parts.append(o[0])
        lses.append(l[0])
    parts, lses = np.stack(parts), np.stack(lses)
    for h in range(2):
        o, l = orc.merge(parts[:, h], lses[:, h])
        np.testing.assert_allclose(o, out[0, h], rtol=1e-12, atol=1e-12)
        assert abs(l - lse[0, h]) < 1e-12
    # empty splits do not change anything; all-empty gives 0 / -inf
    o, l = orc.merge(np.vstack([parts[:, 0], np.zeros((2, 512))]),
                     np.concatenate([lses[:, 0], [-np.inf, -np.inf]]))
    np.testing.assert_allclose(o, out[0, 0], rtol=1e-12, atol=1e-12)
    o, l = orc.merge(np.zeros((3, 512)), np.full(3, -np.inf))
    assert np.all(o == 0) and l == -np.inf


# ---------------------------------------------------------------- cross-API identities

def _ds_cache_from_records(recs: np.ndarray, block_size: int):
    n = recs.shape[0]
    nb = (n + block_size - 1) // block_size
    cache = np.zeros((nb, block_size, 656), dtype=np.uint8)
    cache.reshape(-1, 656)[:n] = recs
    return cache


def test_sparse_equals_paged_decode_on_same_records(orc):
    rng = np.random.default_rng(17)
    B, bs = 3, 16
    case = synth.paged_case(17, synth.DS_MLA, B=B, q_len=1, H=4, L_lo=1, L_hi=70, block_size=bs)
    out_p, lse_p = orc.paged_decode(synth.DS_MLA, case.q, case.cache, case.block_table,
                                    case.seq_lens, 1, case.softmax_scale)
    flat = case.cache.reshape(-1, 656)
    ptr, idx = [0], []
    for b in range(B):
        L = int(case.seq_lens[b])
        p = np.arange(L)
        idx.extend(case.block_table[b, p // bs] * bs + p % bs)
        ptr.append(len(idx))
    q16 = case.q.view(np.uint16)
    out_s, lse_s = orc.sparse_fwd(q16, flat, ptr, idx, case.softmax_scale, False)
    np.testing.assert_allclose(out_s, out_p, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse_s, lse_p, rtol=1e-13, atol=1e-13)


def test_ds_mla_equals_bf16_when_scales_are_powers_of_two(orc):
    rng = np.random.default_rng(23)
    B, bs = 2, 8
    case = synth.paged_case(23, synth.DS_MLA, B=B, q_len=1, H=3, L_lo=5, L_hi=40, block_size=bs)
    flat = case.cache.reshape(-1, 656)
    flat[:, 512:528] = (2.0 ** rng.integers(-4, 5, size=(flat.shape[0], 4))).astype(np.float32).view(np.uint8)
    dec = decoded_ds(flat)
    bf = bf16_bits(dec)
    assert np.array_equal(torch.from_numpy(bf.view(np.int16)).view(torch.bfloat16).double().numpy(), dec)
    cache_bf = bf.view(np.uint8).reshape(case.cache.shape[0], bs, 1152)
    o1, l1 = orc.paged_decode(synth.DS_MLA, case.q, case.cache, case.block_table, case.seq_lens, 1, 0.2)
    o2, l2 = orc.paged_decode(synth.BF16, case.q, cache_bf, case.block_table, case.seq_lens, 1, 0.2)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


def test_fp8_scale_algebra_against_bf16(orc):
    # with q_scale = k_scale = 2, the scaled e4m3 values are exact in bf16
    case = synth.paged_case(29, synth.FP8, B=2, q_len=1, H=2, L_lo=3, L_hi=30, block_size=4,
                            q_scale=2.0, k_scale=2.0)
    cache_vals = torch.from_numpy(case.cache.reshape(-1, 576).copy()).view(torch.float8_e4m3fn).double() * 2.0
    q_vals = torch.from_numpy(case.q.copy()).view(torch.float8_e4m3fn).double() * 2.0
    cache_bf = bf16_bits(cache_vals.numpy()).view(np.uint8).reshape(case.cache.shape[0], 4, 1152)
    q_bf = bf16_bits(q_vals.numpy()).view(np.uint8).reshape(case.q.shape[0], 2, 1152)
    o1, l1 = orc.paged_decode(synth.FP8, case.q, case.cache, case.block_table, case.seq_lens, 1,
                              0.3, q_scale=2.0, k_scale=2.0)
    o2, l2 = orc.paged_decode(synth.BF16, q_bf, cache_bf, case.block_table, case.seq_lens, 1, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


def test_spec_verify_row_equals_shorter_decode(orc):
    qn = 4
    case = synth.paged_case(31, synth.BF16, B=3, q_len=qn, H=2, L_lo=4, L_hi=50, block_size=8)
    out, lse = orc.paged_decode(synth.BF16, case.q, case.cache, case.block_table, case.seq_lens, qn,
                                case.softmax_scale)
    for b in range(3):
        for i in range(qn):
            L1 = np.array([case.seq_lens[b] - qn + 1 + i], dtype=np.int32)
            o1, l1 = orc.paged_decode(synth.BF16, case.q[b * qn + i:b * qn + i + 1], case.cache,
                                      case.block_table[b:b + 1], L1, 1, case.softmax_scale)
            assert np.array_equal(o1[0], out[b * qn + i]) and np.array_equal(l1[0], lse[b * qn + i])


def test_zero_length_request_and_causal_underflow(orc):
    case = synth.paged_case(37, synth.BF16, B=3, q_len=2, H=2, L_lo=1, L_hi=10, block_size=4,
                            seq_lens=[0, 1, 5])
    out, lse = orc.paged_decode(synth.BF16, case.q, case.cache, case.block_table, case.seq_lens, 2, 0.5)
    # request 0 (L = 0): both rows empty; request 1 (L = 1, q = 2): row 0 sees nothing, row 1 key 0
    assert np.all(out[0:3] == 0) and np.all(np.isneginf(lse[0:3]))
    assert np.all(np.isfinite(lse[3:]))


def test_block_id_out_of_range_is_an_error(orc):
    case = synth.paged_case(41, synth.BF16, B=1, q_len=1, H=1, L_lo=9, L_hi=9, block_size=4)
    bt = case.block_table.copy()
    bt[0, 1] = case.cache.shape[0]
    with pytest.raises(ValueError):
        orc.paged_decode(synth.BF16, case.q, case.cache, bt, case.seq_lens, 1, 0.5)
