"""GPU parity of the chunked-context pieces against the fp64 oracle: mla_gather_context
(bit-exact, all three cache formats, bf16 up-convert and stored bytes, chunk offsets, empty
requests, unaligned destinations, bad block ids) and mla_merge_attn_states (within one bf16
rounding of the exact merge; empty sides; strided partials)."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import bf16_bits, t_bf16, t_i32, t_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def chunk_of(case, rng):
    L = case.seq_lens.astype(np.int64)
    starts = np.array([rng.integers(0, max(l, 1)) for l in L], dtype=np.int64)
    lens = np.array([rng.integers(0, l - s + 1) if l > s else 0 for l, s in zip(L, starts)], dtype=np.int64)
    lens[1] = 0                                                     # an empty request inside the chunk
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cu, starts.astype(np.int32)


@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP8, synth.DS_MLA])
@pytest.mark.parametrize("raw", [False, True])
@pytest.mark.parametrize("bs", [16, 64])
def test_gather_bit_exact(m, fmt, raw, bs):
    case = synth.paged_case(870 + fmt + bs, fmt, B=6, q_len=1, H=1, L_lo=50, L_hi=900, block_size=bs,
                            q_scale=0.05, k_scale=0.05)
    cu, starts = chunk_of(case, np.random.default_rng(fmt + bs))
    n = int(cu[-1]) + 5                                             # rows past the chunk stay untouched
    ref = oracle.gather_context(fmt, case.cache, case.block_table, cu, starts, num_tokens=n, raw=raw,
                                scale=case.k_scale)
    dst = m.gather_context(t_u8(case.cache), t_i32(case.block_table), t_i32(cu), t_i32(starts), fmt=fmt,
                           num_tokens=n, raw=raw, scale=case.k_scale)
    got = dst.cpu().numpy() if raw else bf16_bits(dst)
    assert np.array_equal(got[:cu[-1]], ref[:cu[-1]])
    assert m.read_device_errors() == 0


@pytest.mark.parametrize("fmt", [synth.FP8, synth.DS_MLA])
def test_gather_unaligned_rows_and_padded_pitch(m, fmt):
    case = synth.paged_case(880 + fmt, fmt, B=3, q_len=1, H=1, L_lo=40, L_hi=300, block_size=16, entry_pad=16,
                            k_scale=0.03)
    cu = np.concatenate([[0], np.cumsum(case.seq_lens)]).astype(np.int32)
    ref = oracle.gather_context(fmt, case.cache, case.block_table, cu, None, scale=case.k_scale)
    big = torch.zeros((int(cu[-1]), 577), dtype=torch.bfloat16, device="cuda")      # rows 1154 bytes apart
    m.gather_context(t_u8(case.cache), t_i32(case.block_table), t_i32(cu), None, fmt=fmt, num_tokens=int(cu[-1]),
                     scale=case.k_scale, dst=big[:, :576])
    assert np.array_equal(bf16_bits(big[:, :576]), ref) and torch.all(big[:, 576] == 0)


def test_gather_bad_block_gives_zeros_and_flag(m):
    case = synth.paged_case(890, synth.DS_MLA, B=2, q_len=1, H=1, L_lo=100, L_hi=200, block_size=64)
    bt = case.block_table.copy()
    bt[1, 0] = case.cache.shape[0] + 7
    cu = np.array([0, 10, 20], dtype=np.int32)
    m.read_device_errors()
    dst = m.gather_context(t_u8(case.cache), t_i32(bt), t_i32(cu), None, fmt=synth.DS_MLA, num_tokens=20)
    assert m.read_device_errors() & 2
    assert torch.all(dst[10:] == 0)
    ref = oracle.gather_context(synth.DS_MLA, case.cache, case.block_table, cu[:2], None)
    assert np.array_equal(bf16_bits(dst[:10]), ref)


def merge_inputs(seed, T, H, D, empty_p=(), empty_s=(), both=()):
    rng = np.random.default_rng(seed)
    a = synth.normal_bf16_bits(rng, (T, H, D))
    b = synth.normal_bf16_bits(rng, (T, H, D))
    lp = (rng.standard_normal((H, T)) * 6).astype(np.float32)
    ls = (rng.standard_normal((H, T)) * 6).astype(np.float32)
    for t in empty_p:
        lp[:, t] = -np.inf
    for t in empty_s:
        ls[:, t] = -np.inf
    for t in both:
        lp[:, t] = ls[:, t] = -np.inf
    return a, lp, b, ls


def check_merge(out, lse, ref, rl, a, b):
    fa = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()
    fb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()
    o = out.double().cpu().numpy()
    # one bf16 rounding of the fp32 result, plus fp32 error of the weights
    assert np.all(np.abs(o - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * (np.abs(fa) + np.abs(fb)) + 1e-30)
    l = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l), fin) and np.all(l[~fin] == -np.inf)
    assert np.all(np.abs(l[fin] - rl[fin]) <= 1e-5 * (1 + np.abs(rl[fin])))


@pytest.mark.parametrize("D", [128, 512, 100])
def test_merge_states(m, D):
    T, H = 37, 16
    a, lp, b, ls = merge_inputs(900 + D, T, H, D, empty_p=(3,), empty_s=(5,), both=(7,))
    ref, rl = oracle.merge_attn_states(a, lp, b, ls)
    out, lse = m.merge_attn_states(t_bf16(a), torch.from_numpy(lp).cuda(), t_bf16(b), torch.from_numpy(ls).cuda(),
                                   return_lse=True)
    check_merge(out, lse, ref, rl, a, b)
    assert torch.all(out[7] == 0)


def test_merge_strided_partials(m):
    T, H, D = 20, 8, 128
    a, lp, b, ls = merge_inputs(950, T, H, D)
    pa = torch.zeros((T, H, 192), dtype=torch.bfloat16, device="cuda")    # context output padded to 192
    pa[:, :, :D] = t_bf16(a)
    ref, rl = oracle.merge_attn_states(a, lp, b, ls)
    out = torch.full((T, H * D + 8), 3.0, dtype=torch.bfloat16, device="cuda")
    o3 = out[:, :H * D].view(T, H, D)
    m.merge_attn_states(pa[:, :, :D], torch.from_numpy(lp).cuda(), t_bf16(b), torch.from_numpy(ls).cuda(), output=o3)
    _, lse = m.merge_attn_states(pa[:, :, :D], torch.from_numpy(lp).cuda(), t_bf16(b), torch.from_numpy(ls).cuda(),
                                 return_lse=True)
    check_merge(o3, lse, ref, rl, a, b)
    assert torch.all(out[:, H * D:] == 3.0)
