"""Pins of the oracle's decode epilogue (q concat + latent insert) against library casts
(torch CPU bfloat16 / float8_e4m3fn), an fp64 rotation, and the insert's round-trip bounds."""
import numpy as np
import pytest
import torch

from mla_latent_cache_attention_gb300 import synth


def t_bf16(bits) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def make(fmt, B=5, H=3, bs=4, nb=6, seed=0, rope=True, entry_pad=0):
    rng = np.random.default_rng(seed)
    eb = synth.ENTRY_BYTES[fmt]
    cache = np.zeros((nb, bs, eb + entry_pad), dtype=np.uint8)
    slots = rng.choice(nb * bs, size=B, replace=False).astype(np.int64)
    pos = rng.integers(0, 4096, size=B).astype(np.int64)
    epi = synth.epilogue_inputs(seed, B, H, slots, pos, max_position=4096)
    if not rope:
        epi.positions, epi.cos_sin = None, None
    return cache, epi


def run(orc, fmt, cache, epi, **kw):
    return orc.q_concat_cache_insert(fmt, epi.ql_nope, epi.q_pe, epi.kv_c, epi.k_pe, cache,
                                     epi.slot_mapping, positions=epi.positions,
                                     cos_sin=epi.cos_sin, **kw)


def rope64(x: np.ndarray, cs_row: np.ndarray) -> np.ndarray:
    """fp64 GPT-J rotation, for the 1-ulp check."""
    x = x.astype(np.float64)
    c, s = cs_row[:32].astype(np.float64), cs_row[32:].astype(np.float64)
    y = np.empty(64)
    y[0::2] = x[0::2] * c - x[1::2] * s
    y[1::2] = x[1::2] * c + x[0::2] * s
    return y


def test_rope_position_zero_is_identity(orc):
    cs = synth.cos_sin_table(8)
    x = t_bf16(synth.normal_bf16_bits(np.random.default_rng(0), 64)).float().numpy()
    assert np.array_equal(orc.rope_fp32(x, cs[0]), x)


def test_rope_matches_fp64_and_preserves_pair_norms(orc):
    cs = synth.cos_sin_table(131072)
    rng = np.random.default_rng(1)
    for p in rng.integers(0, 131072, 50):
        x = rng.standard_normal(64).astype(np.float32)
        y = orc.rope_fp32(x, cs[p]).astype(np.float64)
        ref = rope64(x, cs[p])
        assert np.max(np.abs(y - ref)) <= 4e-7 * (1 + np.abs(ref)).max()
        n0 = x[0::2].astype(np.float64) ** 2 + x[1::2].astype(np.float64) ** 2
        n1 = y[0::2] ** 2 + y[1::2] ** 2
        np.testing.assert_allclose(n1, n0, rtol=2e-6)
    # rotating by p then by -p (sin negated) gives the input back within fp32 rounding
    x = rng.standard_normal(64).astype(np.float32)
    row = cs[12345].copy()
    inv = row.copy()
    inv[32:] = -inv[32:]
    np.testing.assert_allclose(orc.rope_fp32(orc.rope_fp32(x, row), inv), x, atol=2e-6)


def test_bf16_concat_and_insert(orc):
    cache, epi = make(synth.BF16)
    mqa = run(orc, synth.BF16, cache, epi)
    assert np.array_equal(mqa[:, :, :512], epi.ql_nope)
    B, H = epi.ql_nope.shape[:2]
    for b in range(B):
        cs = epi.cos_sin[epi.positions[b]]
        for h in range(H):
            x = t_bf16(epi.q_pe[b, h]).float().numpy()
            got = t_bf16(mqa[b, h, 512:]).double().numpy()
            ref = rope64(x, cs)
            # one rounding to bf16 from a value within fp32 ulps of the exact rotation
            assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
            assert np.array_equal(mqa[b, h, 512:], bits_of(torch.from_numpy(orc.rope_fp32(x, cs)).to(torch.bfloat16)))
        s = epi.slot_mapping[b]
        ent = cache[s // 4, s % 4]
        assert np.array_equal(ent[:1024].view(np.uint16), epi.kv_c[b])
        kp = orc.rope_fp32(t_bf16(epi.k_pe[b]).float().numpy(), cs)
        assert np.array_equal(ent[1024:].view(np.uint16), bits_of(torch.from_numpy(kp).to(torch.bfloat16)))
    # every other entry stays zero
    touched = np.zeros(cache.shape[:2], dtype=bool)
    touched.reshape(-1)[epi.slot_mapping] = True
    assert np.all(cache[~touched] == 0)


def test_no_rope_copies_bits(orc):
    cache, epi = make(synth.BF16, rope=False)
    mqa = run(orc, synth.BF16, cache, epi)
    assert np.array_equal(mqa[:, :, 512:], epi.q_pe)
    for b, s in enumerate(epi.slot_mapping):
        assert np.array_equal(cache[s // 4, s % 4, 1024:].view(np.uint16), epi.k_pe[b])


def test_fp8_concat_and_insert_match_library_quant(orc):
    cache, epi = make(synth.FP8)
    qinv, cinv = np.float32(1 / 0.05), np.float32(1 / 0.07)
    mqa = run(orc, synth.FP8, cache, epi, q_scale_inv=float(qinv), cache_scale_inv=float(cinv))
    sat = lambda v: torch.from_numpy(np.clip(v, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    B, H = epi.ql_nope.shape[:2]
    for b in range(B):
        cs = epi.cos_sin[epi.positions[b]]
        for h in range(H):
            qn = t_bf16(epi.ql_nope[b, h]).float().numpy()
            assert np.array_equal(mqa[b, h, :512], sat(qn * qinv))   # fp32 product, then quant
            qp = orc.rope_fp32(t_bf16(epi.q_pe[b, h]).float().numpy(), cs)
            assert np.array_equal(mqa[b, h, 512:], sat(qp * qinv))
        s = epi.slot_mapping[b]
        ent = cache[s // 4, s % 4]
        kc = t_bf16(epi.kv_c[b]).float().numpy()
        assert np.array_equal(ent[:512], sat(kc * cinv))
        kp = orc.rope_fp32(t_bf16(epi.k_pe[b]).float().numpy(), cs)
        assert np.array_equal(ent[512:], sat(kp * cinv))
        # round trip: within half an e4m3 ulp of x * inv (values stay below 448)
        dec = torch.from_numpy(ent.copy()).view(torch.float8_e4m3fn).double().numpy()
        x = np.concatenate([kc, kp]).astype(np.float64) * float(cinv)
        ulp = np.where(np.abs(x) < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 1e-30))) - 3))
        assert np.all(np.abs(dec - x) <= ulp / 2 + 1e-12)


def test_ds_mla_insert_scales_and_codes(orc):
    cache, epi = make(synth.DS_MLA, seed=3)
    # widen the dynamic range of one tile per token to exercise the exponent rule
    epi.kv_c = epi.kv_c.copy()
    big = torch.tensor([300.0, -9000.0, 0.001, 57344.0, 7.0]).to(torch.bfloat16)
    for b in range(epi.kv_c.shape[0]):
        epi.kv_c[b, 128 * (b % 4) + 5] = bits_of(big[b % 5:b % 5 + 1])[0]
    mqa = run(orc, synth.DS_MLA, cache, epi)
    assert mqa.dtype == np.uint16 and np.array_equal(mqa[:, :, :512], epi.ql_nope)
    for b in range(epi.kv_c.shape[0]):
        s = epi.slot_mapping[b]
        ent = cache[s // 4, s % 4]
        scales = ent[512:528].copy().view(np.float32).astype(np.float64)
        x = t_bf16(epi.kv_c[b]).double().numpy()
        for j in range(4):
            tile = x[128 * j:128 * (j + 1)]
            amax = np.abs(tile).max()
            sj = scales[j]
            k = int(np.log2(sj))
            assert sj == 2.0 ** k                                  # a power of two
            assert amax <= 448 * sj and amax > 224 * sj            # smallest such power
            codes = ent[128 * j:128 * (j + 1)]
            ref = torch.from_numpy((tile / sj).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(codes, ref)
        kp = orc.rope_fp32(t_bf16(epi.k_pe[b]).float().numpy(), epi.cos_sin[epi.positions[b]])
        assert np.array_equal(ent[528:].view(np.uint16), bits_of(torch.from_numpy(kp).to(torch.bfloat16)))


def test_ds_mla_zero_tile_gets_unit_scale(orc):
    cache, epi = make(synth.DS_MLA, B=1, seed=4)
    epi.kv_c = epi.kv_c.copy()
    epi.kv_c[0, 256:384] = 0
    run(orc, synth.DS_MLA, cache, epi)
    s = epi.slot_mapping[0]
    ent = cache[s // 4, s % 4]
    assert ent[512 + 8:512 + 12].view(np.float32)[0] == 1.0 and np.all(ent[256:384] == 0)


def test_negative_slot_skips_insert_but_writes_query(orc):
    cache, epi = make(synth.BF16, seed=5)
    epi.slot_mapping = epi.slot_mapping.copy()
    epi.slot_mapping[1] = -1
    mqa = run(orc, synth.BF16, cache, epi)
    assert np.array_equal(mqa[1, :, :512], epi.ql_nope[1])
    assert int((cache.reshape(-1, 1152).any(axis=1)).sum()) == epi.slot_mapping.size - 1


def test_padded_entry_stride(orc):
    cache, epi = make(synth.DS_MLA, seed=6, entry_pad=16)
    cache2, _ = make(synth.DS_MLA, seed=6)
    run(orc, synth.DS_MLA, cache, epi)
    run(orc, synth.DS_MLA, cache2, epi)
    assert np.array_equal(cache[:, :, :656], cache2) and np.all(cache[:, :, 656:] == 0)


def test_positions_without_table_is_an_error(orc):
    cache, epi = make(synth.BF16)
    with pytest.raises(ValueError):
        orc.q_concat_cache_insert(synth.BF16, epi.ql_nope, epi.q_pe, epi.kv_c, epi.k_pe, cache,
                                  epi.slot_mapping, positions=epi.positions, cos_sin=None)
