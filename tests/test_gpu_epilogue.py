"""GPU parity of the decode epilogue (q concat + latent insert): bit-exact against the oracle
for all three cache formats, with and without RoPE, padded entry pitch, skipped slots."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import bf16_bits, t_bf16, t_i64, t_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def run_both(m, fmt, B, H, bs, nb, seed, rope=True, entry_pad=0, neg_slot=False, wide=False):
    rng = np.random.default_rng(seed)
    eb = synth.ENTRY_BYTES[fmt]
    cache = rng.integers(0, 256, size=(nb, bs, eb + entry_pad), dtype=np.uint8)   # stale bytes
    if fmt == synth.DS_MLA:
        cache[:, :, 512:528] = 0
    slots = rng.choice(nb * bs, size=B, replace=False).astype(np.int64)
    if neg_slot:
        slots[::3] = -1
    pos = rng.integers(0, 4096, size=B)
    epi = synth.epilogue_inputs(seed, B, H, slots, pos, max_position=4096)
    if wide:   # per-tile dynamic range: huge, tiny, zero tiles
        kv = epi.kv_c.copy()
        f = torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16).float()
        f[:, 0:128] *= 3000.0
        f[:, 128:256] *= 1e-5
        f[::2, 256:384] = 0.0
        epi.kv_c = f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qinv, cinv = np.float32(1 / 0.05), np.float32(1 / 0.03)
    kw = {}
    if fmt == synth.FP8:
        kw = dict(q_scale_inv=float(qinv), cache_scale_inv=float(cinv))
    ref_cache = cache.copy()
    ref_q = oracle.q_concat_cache_insert(fmt, epi.ql_nope, epi.q_pe, epi.kv_c, epi.k_pe, ref_cache, slots,
                                         positions=epi.positions if rope else None,
                                         cos_sin=epi.cos_sin if rope else None, **kw)
    gcache = t_u8(cache)
    gkw = {}
    if fmt == synth.FP8:
        gkw = dict(q_scale_inv=torch.tensor([qinv], device="cuda"), cache_scale_inv=torch.tensor([cinv], device="cuda"))
    gq = m.q_concat_cache_insert(t_bf16(epi.ql_nope), t_bf16(epi.q_pe), t_bf16(epi.kv_c), t_bf16(epi.k_pe), gcache,
                                 t_i64(slots), fmt=fmt, positions=t_i64(epi.positions) if rope else None,
                                 cos_sin_cache=torch.from_numpy(epi.cos_sin).cuda() if rope else None, **gkw)
    torch.cuda.synchronize()
    if fmt == synth.FP8:
        assert np.array_equal(gq.cpu().numpy(), ref_q)
    else:
        assert np.array_equal(bf16_bits(gq), ref_q)
    assert np.array_equal(gcache.cpu().numpy(), ref_cache)
    assert m.read_device_errors() == 0


@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP8, synth.DS_MLA])
@pytest.mark.parametrize("rope", [True, False])
def test_epilogue_bit_exact(m, fmt, rope):
    run_both(m, fmt, B=37, H=16, bs=8, nb=20, seed=fmt * 10 + rope, rope=rope)


@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP8, synth.DS_MLA])
def test_epilogue_padded_pitch_skipped_slots_odd_heads(m, fmt):
    run_both(m, fmt, B=19, H=5, bs=16, nb=4, seed=50 + fmt, entry_pad=48, neg_slot=True)


def test_ds_mla_insert_wide_dynamic_range(m):
    run_both(m, synth.DS_MLA, B=24, H=3, bs=4, nb=10, seed=77, wide=True)


def test_epilogue_config1_shape(m):
    case, epi = synth.config1()
    cache = case.cache.copy()
    ref_q = oracle.q_concat_cache_insert(synth.BF16, epi.ql_nope, epi.q_pe, epi.kv_c, epi.k_pe, cache,
                                         epi.slot_mapping, positions=epi.positions, cos_sin=epi.cos_sin)
    gcache = t_u8(case.cache)
    gq = m.q_concat_cache_insert(t_bf16(epi.ql_nope), t_bf16(epi.q_pe), t_bf16(epi.kv_c), t_bf16(epi.k_pe), gcache,
                                 t_i64(epi.slot_mapping), fmt=synth.BF16, positions=t_i64(epi.positions),
                                 cos_sin_cache=torch.from_numpy(epi.cos_sin).cuda())
    assert np.array_equal(bf16_bits(gq), ref_q)
    assert np.array_equal(gcache.cpu().numpy(), cache)


def test_bad_slot_and_position_are_flagged(m):
    case, epi = synth.config1(B=4, L_lo=10, L_hi=20)
    gcache = t_u8(case.cache)
    slots = epi.slot_mapping.copy()
    slots[1] = case.cache.shape[0] * 64 + 5          # block beyond the pool
    pos = epi.positions.copy()
    pos[2] = 10 ** 7                                 # beyond the table
    m.read_device_errors()
    m.q_concat_cache_insert(t_bf16(epi.ql_nope), t_bf16(epi.q_pe), t_bf16(epi.kv_c), t_bf16(epi.k_pe), gcache,
                            t_i64(slots), fmt=synth.BF16, positions=t_i64(pos),
                            cos_sin_cache=torch.from_numpy(epi.cos_sin).cuda())
    flags = m.read_device_errors()
    assert flags & 4 and flags & 8
