"""GPU parity of the per-head contractions around the attention core against the fp64 oracle:
mla_absorb_q (BMM1 with W_UK_T) and mla_v_up_proj (W_UV, with and without the sigmoid output
gate), over decode batch sizes that are not multiples of the 64-token tile, 16 and 96 heads,
strided and unaligned inputs; and the whole absorbed decode layer (BMM1 -> epilogue -> paged
decode -> W_UV + gate) on synthetic weights."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import bf16_bits, t_bf16, t_i32, t_i64, t_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def weights(rng, H, K, F):
    """bf16 [H, K, F] ~ N(0, 1/K): unit-scale outputs for unit-scale inputs."""
    w = rng.standard_normal((H, K, F)).astype(np.float32) / np.sqrt(K)
    return torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def check(got_bits, x, w, exact, gate_terms=1):
    """One bf16 rounding per step (the product, and with a gate the gate and the gated value),
    plus fp32 accumulation: |gpu - exact| <= 2^-8 (steps) |exact| + 2^-16 sum_k |x w|."""
    mag = np.einsum("bhk,hkf->bhf", np.abs(f64(x)), np.abs(f64(w)))
    got = f64(got_bits)
    err = np.abs(got - exact)
    bound = 2.0 ** -8 * gate_terms * np.abs(exact) + 2.0 ** -16 * mag
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"


@pytest.mark.parametrize("B,H", [(1, 16), (32, 16), (100, 96), (128, 96)])
def test_absorb_q(m, B, H):
    rng = np.random.default_rng(B + H)
    q = synth.normal_bf16_bits(rng, (B, H, 192))            # [q_nope (128) | q_pe (64)]
    w = weights(rng, H, 128, 512)
    ql = m.absorb_q(t_bf16(q)[:, :, :128], t_bf16(w))
    exact = oracle.head_bmm(q[:, :, :128], w)
    check(bf16_bits(ql), q[:, :, :128], w, exact)


def test_absorb_q_unaligned_rows(m):
    rng = np.random.default_rng(5)
    q = synth.normal_bf16_bits(rng, (20, 16, 129))
    w = weights(rng, 16, 128, 512)
    ql = m.absorb_q(t_bf16(q)[:, :, 1:], t_bf16(w))         # rows 2 bytes off the 16-byte grid
    check(bf16_bits(ql), q[:, :, 1:], w, oracle.head_bmm(q[:, :, 1:], w))


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("B,H", [(7, 16), (128, 96)])
def test_v_up_proj(m, gated, B, H):
    rng = np.random.default_rng(10 * B + H + gated)
    lat = synth.normal_bf16_bits(rng, (B, H, 512))
    w = weights(rng, H, 512, 128)
    g = synth.normal_bf16_bits(rng, (B, H * 128)) if gated else None
    out = torch.full((B, H * 128 + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    o3 = out[:, :H * 128].view(B, H, 128)
    m.v_up_proj(t_bf16(lat), t_bf16(w), None if g is None else t_bf16(g), out=o3)
    exact = oracle.head_bmm(lat, w, g)
    check(bf16_bits(o3), lat, w, exact, gate_terms=3 if gated else 1)
    assert torch.all(out[:, H * 128:] == 7.0)


def test_absorbed_decode_layer(m):
    """BMM1 -> decode epilogue (q concat + RoPE + bf16 insert) -> paged decode -> W_UV + gate,
    against the oracle chain fed the GPU's bf16 hand-offs (each stage is pinned separately)."""
    rng = np.random.default_rng(77)
    case, epi = synth.config1(B=8, L_lo=300, L_hi=2000)
    B, H = 8, 16
    q_nope = synth.normal_bf16_bits(rng, (B, H, 128))
    w_uk = weights(rng, H, 128, 512)
    w_uv = weights(rng, H, 512, 128)
    gate = synth.normal_bf16_bits(rng, (B, H * 128))
    gcache = t_u8(case.cache)
    ql = m.absorb_q(t_bf16(q_nope), t_bf16(w_uk))
    mqa = m.q_concat_cache_insert(ql, t_bf16(epi.q_pe), t_bf16(epi.kv_c), t_bf16(epi.k_pe), gcache,
                                  t_i64(epi.slot_mapping), fmt=synth.BF16, positions=t_i64(epi.positions),
                                  cos_sin_cache=torch.from_numpy(epi.cos_sin).cuda())
    lat, _ = m.paged_decode(mqa, gcache, t_i32(case.block_table), t_i32(case.seq_lens), fmt=synth.BF16,
                            max_context=case.max_context, softmax_scale=case.softmax_scale)
    out = m.v_up_proj(lat, t_bf16(w_uv), t_bf16(gate))
    # oracle chain
    check(bf16_bits(ql), q_nope, w_uk, oracle.head_bmm(q_nope, w_uk))
    cache = case.cache.copy()
    ref_q = oracle.q_concat_cache_insert(synth.BF16, bf16_bits(ql), epi.q_pe, epi.kv_c, epi.k_pe, cache,
                                         epi.slot_mapping, positions=epi.positions, cos_sin=epi.cos_sin)
    assert np.array_equal(bf16_bits(mqa), ref_q)
    ro, _ = oracle.paged_decode(synth.BF16, ref_q.view(np.uint8).reshape(B, H, 1152), cache, case.block_table,
                                case.seq_lens, 1, case.softmax_scale)
    o = lat.double().cpu().numpy()
    assert np.all(np.abs(o - ro) <= 1e-2 + 1e-2 * np.abs(ro))
    check(bf16_bits(out), bf16_bits(lat), w_uv, oracle.head_bmm(bf16_bits(lat), w_uv, gate), gate_terms=3)
    assert m.read_device_errors() == 0
