"""GPU parity of the prefill epilogues (mla_key_concat_cache_insert for the bf16 and
fp8_ds_mla caches, mla_qkv_quant_cache_fp8_insert for the plain fp8 cache) against the fp64
oracle: bit-exact k_out, rotated q, q/k/v codes and cache bytes, with and without RoPE, with
skipped slots, padded cache pitch, strided inputs and a prefill-sized batch (Tp=4096, H=16)."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import bf16_bits, t_bf16, t_i64, t_u8

pytestmark = pytest.mark.gpu
DN, DV = 128, 128


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def inputs(seed, Tp, H, nb, bs, fmt, rope=True, skip=(), entry_pad=0, max_pos=131072):
    rng = np.random.default_rng(seed)
    g = lambda *shape: synth.normal_bf16_bits(rng, shape)
    d = dict(q=g(Tp, H, DN + 64), k_nope=g(Tp, H, DN), k_pe=g(Tp, 64), kv_c=g(Tp, 512), v=g(Tp, H, DV),
             slots=rng.choice(nb * bs, size=Tp, replace=False).astype(np.int64),
             pos=rng.integers(0, max_pos, size=Tp).astype(np.int64) if rope else None,
             cs=synth.cos_sin_table(max_pos) if rope else None)
    for t in skip:
        d["slots"][t] = -1
    cache = np.zeros((nb, bs, synth.ENTRY_BYTES[fmt] + entry_pad), dtype=np.uint8)
    # stale bytes where nothing is written must survive
    cache[:] = rng.integers(0, 256, size=cache.shape, dtype=np.uint8)
    return d, cache


def dev_rope(d):
    if d["pos"] is None:
        return None, None
    return t_i64(d["pos"]), torch.from_numpy(d["cs"]).cuda()


@pytest.mark.parametrize("fmt", [synth.BF16, synth.DS_MLA])
@pytest.mark.parametrize("rope", [True, False])
def test_key_concat_bit_exact(m, fmt, rope):
    d, cache = inputs(40 + fmt + 2 * rope, Tp=37, H=20, nb=12, bs=16, fmt=fmt, rope=rope, skip=(3, 30))
    ref_cache = cache.copy()
    ref_q = d["q"].copy()
    ref_k = oracle.key_concat_cache_insert(fmt, ref_q, d["k_nope"], d["k_pe"], d["kv_c"], ref_cache, d["slots"],
                                           positions=d["pos"], cos_sin=d["cs"])
    q, gcache = t_bf16(d["q"]), t_u8(cache)
    pos, cs = dev_rope(d)
    k_out = m.key_concat_cache_insert(q, t_bf16(d["k_nope"]), t_bf16(d["k_pe"]), t_bf16(d["kv_c"]), gcache,
                                      t_i64(d["slots"]), fmt=fmt, positions=pos, cos_sin_cache=cs)
    assert np.array_equal(bf16_bits(k_out), ref_k)
    assert np.array_equal(bf16_bits(q), ref_q)
    assert np.array_equal(gcache.cpu().numpy(), ref_cache)
    assert m.read_device_errors() == 0


def test_key_concat_strided_inputs_and_padded_pitch(m):
    fmt = synth.DS_MLA
    d, cache = inputs(47, Tp=9, H=5, nb=4, bs=8, fmt=fmt, entry_pad=16)
    ref_cache, ref_q = cache.copy(), d["q"].copy()
    ref_k = oracle.key_concat_cache_insert(fmt, ref_q, d["k_nope"], d["k_pe"], d["kv_c"], ref_cache, d["slots"],
                                           positions=d["pos"], cos_sin=d["cs"])
    qbig = torch.zeros((9, 5, 200), dtype=torch.bfloat16, device="cuda")
    qbig[:, :, :192] = t_bf16(d["q"])
    knbig = torch.zeros((9, 5, 136), dtype=torch.bfloat16, device="cuda")
    knbig[:, :, 3:131] = t_bf16(d["k_nope"])               # unaligned rows: the scalar path
    gcache = t_u8(cache)
    pos, cs = dev_rope(d)
    k_out = m.key_concat_cache_insert(qbig[:, :, :192], knbig[:, :, 3:131], t_bf16(d["k_pe"]), t_bf16(d["kv_c"]),
                                      gcache, t_i64(d["slots"]), fmt=fmt, positions=pos, cos_sin_cache=cs)
    assert np.array_equal(bf16_bits(k_out), ref_k)
    assert np.array_equal(bf16_bits(qbig[:, :, :192]), ref_q)
    assert torch.all(qbig[:, :, 192:] == 0)
    assert np.array_equal(gcache.cpu().numpy(), ref_cache)


@pytest.mark.parametrize("rope", [True, False])
def test_qkv_quant_fp8_bit_exact(m, rope):
    d, cache = inputs(50 + rope, Tp=29, H=12, nb=10, bs=16, fmt=synth.FP8, rope=rope, skip=(0,))
    sc = dict(q_scale_inv=1 / 0.05, k_scale_inv=1 / 0.03, v_scale_inv=1 / 0.02, cache_scale_inv=1 / 0.07)
    ref_cache = cache.copy()
    rq, rk, rv = oracle.qkv_quant_cache_fp8_insert(d["q"], d["k_nope"], d["k_pe"], d["kv_c"], d["v"], ref_cache,
                                                   d["slots"], positions=d["pos"], cos_sin=d["cs"],
                                                   **{k: float(np.float32(v)) for k, v in sc.items()})
    gcache = t_u8(cache)
    pos, cs = dev_rope(d)
    q = t_bf16(d["q"])
    dsc = {k: torch.tensor([np.float32(v)], dtype=torch.float32, device="cuda") for k, v in sc.items()}
    q8, k8, v8 = m.qkv_quant_cache_fp8_insert(q, t_bf16(d["k_nope"]), t_bf16(d["k_pe"]), t_bf16(d["kv_c"]),
                                              t_bf16(d["v"]), gcache, t_i64(d["slots"]), positions=pos,
                                              cos_sin_cache=cs, **dsc)
    assert np.array_equal(q8.cpu().numpy(), rq)
    assert np.array_equal(k8.cpu().numpy(), rk)
    assert np.array_equal(v8.cpu().numpy(), rv)
    assert np.array_equal(gcache.cpu().numpy(), ref_cache)
    assert np.array_equal(bf16_bits(q), d["q"])                 # q is only read
    assert m.read_device_errors() == 0


@pytest.mark.parametrize("fmt", [synth.BF16, synth.DS_MLA, synth.FP8])
def test_prefill_sized_batch(m, fmt):
    # Tp = 4096 prefill tokens, H = 16 heads, block_size 64 (the sparse-prefill configuration's
    # sizes); 1024 tokens for fp8, whose oracle encodes every E4M3 value by a search of the grid
    Tp, H = (1024 if fmt == synth.FP8 else 4096), 16
    d, cache = inputs(60 + fmt, Tp=Tp, H=H, nb=80, bs=64, fmt=fmt, skip=(7, Tp - 1))
    ref_cache = cache.copy()
    pos, cs = dev_rope(d)
    gcache = t_u8(cache)
    if fmt == synth.FP8:
        rq, rk, rv = oracle.qkv_quant_cache_fp8_insert(d["q"], d["k_nope"], d["k_pe"], d["kv_c"], d["v"], ref_cache,
                                                       d["slots"], q_scale_inv=1.0, k_scale_inv=1.0, v_scale_inv=1.0,
                                                       cache_scale_inv=20.0, positions=d["pos"], cos_sin=d["cs"])
        one = torch.ones(1, dtype=torch.float32, device="cuda")
        q8, k8, v8 = m.qkv_quant_cache_fp8_insert(t_bf16(d["q"]), t_bf16(d["k_nope"]), t_bf16(d["k_pe"]),
                                                  t_bf16(d["kv_c"]), t_bf16(d["v"]), gcache, t_i64(d["slots"]),
                                                  q_scale_inv=one, k_scale_inv=one, v_scale_inv=one,
                                                  cache_scale_inv=one * 20, positions=pos, cos_sin_cache=cs)
        assert np.array_equal(q8.cpu().numpy(), rq) and np.array_equal(k8.cpu().numpy(), rk)
        assert np.array_equal(v8.cpu().numpy(), rv)
    else:
        ref_q = d["q"].copy()
        ref_k = oracle.key_concat_cache_insert(fmt, ref_q, d["k_nope"], d["k_pe"], d["kv_c"], ref_cache, d["slots"],
                                               positions=d["pos"], cos_sin=d["cs"])
        q = t_bf16(d["q"])
        k_out = m.key_concat_cache_insert(q, t_bf16(d["k_nope"]), t_bf16(d["k_pe"]), t_bf16(d["kv_c"]), gcache,
                                          t_i64(d["slots"]), fmt=fmt, positions=pos, cos_sin_cache=cs)
        assert np.array_equal(bf16_bits(k_out), ref_k) and np.array_equal(bf16_bits(q), ref_q)
    assert np.array_equal(gcache.cpu().numpy(), ref_cache)
    assert m.read_device_errors() == 0


def test_bad_slot_and_position_are_flagged(m):
    d, cache = inputs(70, Tp=4, H=2, nb=2, bs=16, fmt=synth.BF16)
    d["slots"][1] = 2 * 16 + 5                                  # block 2 of 2: out of range
    d["pos"][2] = 10 ** 7                                       # past the table: clamped
    m.read_device_errors()
    pos, cs = dev_rope(d)
    m.key_concat_cache_insert(t_bf16(d["q"]), t_bf16(d["k_nope"]), t_bf16(d["k_pe"]), t_bf16(d["kv_c"]),
                              t_u8(cache), t_i64(d["slots"]), fmt=synth.BF16, positions=pos, cos_sin_cache=cs)
    assert m.read_device_errors() == 4 | 8
