"""Pins of the oracle's prefill epilogues ("vllm.models.kimi_k3.nvidia.ops.
fused_mla_key_concat_kv_cache": fused_mla_key_concat_kv_cache_insert,
fused_mla_key_concat_ds_mla_insert, fused_mla_qkv_quant_kv_cache_fp8_insert) against library
casts (torch CPU bfloat16 / float8_e4m3fn), the fp32 rotation (itself pinned against fp64 in
test_oracle_epilogue.py), the identity at position 0, and the decode epilogue's latent insert
(the same cache entry must come out of both epilogues)."""
import numpy as np
import pytest
import torch

from mla_latent_cache_attention_gb300 import synth

DN, DV = 128, 128


def t_bf16(bits) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sat(v) -> np.ndarray:
    return torch.from_numpy(np.clip(v, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def make(fmt, Tp=6, H=3, bs=4, nb=5, seed=0, rope=True, max_pos=4096):
    rng = np.random.default_rng(seed)
    g = lambda *shape: synth.normal_bf16_bits(rng, shape)
    d = dict(q=g(Tp, H, DN + 64), k_nope=g(Tp, H, DN), k_pe=g(Tp, 64), kv_c=g(Tp, 512), v=g(Tp, H, DV),
             slots=rng.choice(nb * bs, size=Tp, replace=False).astype(np.int64),
             pos=rng.integers(0, max_pos, size=Tp).astype(np.int64) if rope else None,
             cs=synth.cos_sin_table(max_pos) if rope else None)
    cache = np.zeros((nb, bs, synth.ENTRY_BYTES[fmt]), dtype=np.uint8)
    return d, cache


def key_concat(orc, fmt, d, cache):
    q = d["q"].copy()
    k_out = orc.key_concat_cache_insert(fmt, q, d["k_nope"], d["k_pe"], d["kv_c"], cache, d["slots"],
                                        positions=d["pos"], cos_sin=d["cs"])
    return q, k_out


def rot(orc, bits, cs_row):
    return orc.rope_fp32(t_bf16(bits).float().numpy(), cs_row)


@pytest.mark.parametrize("fmt", [synth.BF16, synth.DS_MLA])
def test_key_concat_and_q_rope(orc, fmt):
    d, cache = make(fmt, seed=1)
    q, k_out = key_concat(orc, fmt, d, cache)
    Tp, H = d["k_nope"].shape[:2]
    assert np.array_equal(k_out[:, :, :DN], d["k_nope"])
    assert np.array_equal(q[:, :, :DN], d["q"][:, :, :DN])        # the NoPE part of q is untouched
    for t in range(Tp):
        cs = d["cs"][d["pos"][t]]
        kp = bits_of(torch.from_numpy(rot(orc, d["k_pe"][t], cs)).to(torch.bfloat16))
        for h in range(H):
            assert np.array_equal(k_out[t, h, DN:], kp)           # k_pe broadcast to every head
            qr = bits_of(torch.from_numpy(rot(orc, d["q"][t, h, DN:], cs)).to(torch.bfloat16))
            assert np.array_equal(q[t, h, DN:], qr)


@pytest.mark.parametrize("fmt", [synth.BF16, synth.DS_MLA])
def test_latent_insert_equals_decode_epilogue_insert(orc, fmt):
    d, cache = make(fmt, seed=2)
    key_concat(orc, fmt, d, cache)
    ref = np.zeros_like(cache)
    Tp = d["kv_c"].shape[0]
    ql = np.zeros((Tp, 1, 512), dtype=np.uint16)
    qp = np.zeros((Tp, 1, 64), dtype=np.uint16)
    orc.q_concat_cache_insert(fmt, ql, qp, d["kv_c"], d["k_pe"], ref, d["slots"], positions=d["pos"], cos_sin=d["cs"])
    assert np.array_equal(cache, ref)
    assert int(cache.reshape(-1, cache.shape[2]).any(axis=1).sum()) == Tp


def test_position_zero_and_no_rope_are_identities(orc):
    for rope in (False, True):
        d, cache = make(synth.BF16, seed=3, rope=rope)
        if rope:
            d["pos"] = np.zeros_like(d["pos"])
        q, k_out = key_concat(orc, synth.BF16, d, cache)
        assert np.array_equal(q, d["q"])
        assert np.array_equal(k_out[:, :, DN:], np.broadcast_to(d["k_pe"][:, None, :], k_out[:, :, DN:].shape))
        for t, s in enumerate(d["slots"]):
            ent = cache[s // 4, s % 4]
            assert np.array_equal(ent[:1024].view(np.uint16), d["kv_c"][t])
            assert np.array_equal(ent[1024:].view(np.uint16), d["k_pe"][t])


def test_ds_mla_prefill_insert_scales(orc):
    d, cache = make(synth.DS_MLA, seed=4)
    key_concat(orc, synth.DS_MLA, d, cache)
    for t, s in enumerate(d["slots"]):
        ent = cache[s // 4, s % 4]
        x = t_bf16(d["kv_c"][t]).double().numpy()
        for j in range(4):
            tile, sj = x[128 * j:128 * (j + 1)], float(ent[512 + 4 * j:516 + 4 * j].view(np.float32)[0])
            assert sj == 2.0 ** int(np.log2(sj)) and 224 * sj < np.abs(tile).max() <= 448 * sj
            assert np.array_equal(ent[128 * j:128 * (j + 1)], sat(tile / sj))


def test_negative_slot_skips_insert(orc):
    d, cache = make(synth.BF16, seed=5)
    d["slots"] = d["slots"].copy()
    d["slots"][2] = -1
    _, k_out = key_concat(orc, synth.BF16, d, cache)
    assert int(cache.reshape(-1, 1152).any(axis=1).sum()) == d["slots"].size - 1
    assert np.array_equal(k_out[2, :, :DN], d["k_nope"][2])


def test_fp8_qkv_quant_matches_library_quant(orc):
    d, cache = make(synth.FP8, seed=6)
    qi, ki, vi, ci = np.float32(1 / 0.05), np.float32(1 / 0.03), np.float32(1 / 0.02), np.float32(1 / 0.07)
    q_in = d["q"].copy()
    q8, k8, v8 = orc.qkv_quant_cache_fp8_insert(d["q"], d["k_nope"], d["k_pe"], d["kv_c"], d["v"], cache,
                                                d["slots"], q_scale_inv=qi, k_scale_inv=ki, v_scale_inv=vi,
                                                cache_scale_inv=ci, positions=d["pos"], cos_sin=d["cs"])
    assert np.array_equal(d["q"], q_in)                                  # q is not modified
    Tp, H = d["k_nope"].shape[:2]
    f = lambda bits: t_bf16(bits).float().numpy()
    for t in range(Tp):
        cs = d["cs"][d["pos"][t]]
        kp = rot(orc, d["k_pe"][t], cs)
        for h in range(H):
            assert np.array_equal(q8[t, h, :DN], sat(f(d["q"][t, h, :DN]) * qi))   # fp32 product, then quant
            assert np.array_equal(q8[t, h, DN:], sat(rot(orc, d["q"][t, h, DN:], cs) * qi))
            assert np.array_equal(k8[t, h, :DN], sat(f(d["k_nope"][t, h]) * ki))
            assert np.array_equal(k8[t, h, DN:], sat(kp * ki))
            assert np.array_equal(v8[t, h], sat(f(d["v"][t, h]) * vi))
    # the cache takes its own scale: the same entry as the decode epilogue's fp8 insert
    ref = np.zeros_like(cache)
    ql = np.zeros((Tp, 1, 512), dtype=np.uint16)
    qp = np.zeros((Tp, 1, 64), dtype=np.uint16)
    orc.q_concat_cache_insert(synth.FP8, ql, qp, d["kv_c"], d["k_pe"], ref, d["slots"], q_scale_inv=1.0,
                              cache_scale_inv=float(ci), positions=d["pos"], cos_sin=d["cs"])
    assert np.array_equal(cache, ref)


def test_fp8_scales_are_separate(orc):
    d, c1 = make(synth.FP8, seed=7)
    _, c2 = make(synth.FP8, seed=7)
    a = orc.qkv_quant_cache_fp8_insert(d["q"], d["k_nope"], d["k_pe"], d["kv_c"], d["v"], c1, d["slots"],
                                       q_scale_inv=1.0, k_scale_inv=1.0, v_scale_inv=1.0, cache_scale_inv=4.0,
                                       positions=d["pos"], cos_sin=d["cs"])
    b = orc.qkv_quant_cache_fp8_insert(d["q"], d["k_nope"], d["k_pe"], d["kv_c"], d["v"], c2, d["slots"],
                                       q_scale_inv=1.0, k_scale_inv=2.0, v_scale_inv=1.0, cache_scale_inv=4.0,
                                       positions=d["pos"], cos_sin=d["cs"])
    assert np.array_equal(c1, c2) and np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
    assert not np.array_equal(a[1], b[1])


def test_out_of_range_slot_is_reported(orc):
    d, cache = make(synth.BF16, seed=8)
    d["slots"] = d["slots"].copy()
    d["slots"][0] = 10 ** 6
    with pytest.raises(ValueError):
        key_concat(orc, synth.BF16, d, cache)
