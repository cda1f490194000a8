"""GPU parity of the paged decode / spec-verify against the fp64 oracle: all three cache
formats, q_len 1 and 4 (causal), split-K + merge, zero-length requests, odd block sizes and
head counts; the bf16 decode + epilogue configuration in full, and the fp8 spec-verify
(B=64, q=4, L ~ U[16k, 128k], all 256 query rows) and ds_mla H=96 (B=128, L ~ U[8k, 32k],
all 128 rows) configurations at full size on every row and head."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import (assert_attn_close, assert_lse_close, bf16_bits, t_bf16, t_i32, t_i64, t_u8)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def gpu_q(case):
    if case.fmt == synth.FP8:
        return t_u8(case.q)
    return t_bf16(case.q.view(np.uint16))


def run(m, case, rows=None, max_context=None):
    mc = case.max_context if max_context is None else max_context
    o, l = m.paged_decode(gpu_q(case), t_u8(case.cache), t_i32(case.block_table), t_i32(case.seq_lens),
                          fmt=case.fmt, q_len=case.q_len, max_context=mc, softmax_scale=case.softmax_scale,
                          q_scale=case.q_scale, k_scale=case.k_scale, return_lse=case.return_lse)
    ro, rl = oracle.paged_decode(case.fmt, case.q, case.cache, case.block_table, case.seq_lens, case.q_len,
                                 case.softmax_scale, case.q_scale, case.k_scale, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, device=o.device)
        o = o[idx]
        l = l[idx] if l is not None else None
    return o, l, ro, rl


FMTS = [synth.BF16, synth.FP8, synth.DS_MLA]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("q_len", [1, 4])
def test_small_all_lengths(m, fmt, q_len):
    lens = [0, 1, 3, 127, 128, 129, 300, 1000]
    kw = dict(q_scale=0.05, k_scale=0.05) if fmt == synth.FP8 else {}
    case = synth.paged_case(300 + fmt * 10 + q_len, fmt, B=len(lens), q_len=q_len, H=16, L_lo=1, L_hi=1000,
                            block_size=64, seq_lens=lens, **kw)
    o, l, ro, rl = run(m, case)
    assert_attn_close(o, ro, f"fmt={fmt} q={q_len}")
    assert_lse_close(l, rl, f"fmt={fmt} q={q_len}")


@pytest.mark.parametrize("fmt", FMTS)
def test_split_k_and_merge(m, fmt):
    # a max_context far above the lengths forces several splits per row
    kw = dict(q_scale=0.05, k_scale=0.05) if fmt == synth.FP8 else {}
    case = synth.paged_case(400 + fmt, fmt, B=3, q_len=2, H=16, L_lo=2000, L_hi=9000, block_size=64,
                            max_context=65536, **kw)
    assert m.paged_decode_workspace_size(3, 2, 16, 65536) > 0
    o, l, ro, rl = run(m, case)
    assert_attn_close(o, ro, "split-K")
    assert_lse_close(l, rl, "split-K")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("bs,H", [(1, 16), (16, 3), (32, 20), (64, 96)])
def test_block_sizes_and_heads(m, fmt, bs, H):
    kw = dict(q_scale=0.05, k_scale=0.05) if fmt == synth.FP8 else {}
    case = synth.paged_case(500 + bs + H + fmt, fmt, B=3, q_len=1, H=H, L_lo=50, L_hi=400, block_size=bs, **kw)
    o, l, ro, rl = run(m, case)
    assert_attn_close(o, ro, f"bs={bs} H={H}")
    assert_lse_close(l, rl, f"bs={bs} H={H}")


@pytest.mark.parametrize("fmt,H,q_len", [(synth.BF16, 16, 3), (synth.FP8, 16, 5), (synth.FP8, 128, 1),
                                         (synth.BF16, 128, 2), (synth.FP8, 8, 3), (synth.BF16, 48, 1)])
def test_query_column_groups(m, fmt, H, q_len):
    # query columns (token, head) split into groups: within a token, several tokens per group
    # (with a ragged last group), and a request that fits one group
    kw = dict(q_scale=0.05, k_scale=0.05) if fmt == synth.FP8 else {}
    case = synth.paged_case(700 + H + q_len + fmt, fmt, B=3, q_len=q_len, H=H, L_lo=5, L_hi=1500, block_size=64,
                            max_context=16384, **kw)
    o, l, ro, rl = run(m, case)
    assert_attn_close(o, ro, f"H={H} q_len={q_len}")
    assert_lse_close(l, rl, f"H={H} q_len={q_len}")


def test_padded_entry_pitch(m):
    case = synth.paged_case(601, synth.DS_MLA, B=4, q_len=1, H=16, L_lo=100, L_hi=700, block_size=64,
                            entry_pad=16)
    o, l, ro, rl = run(m, case)
    assert_attn_close(o, ro, "padded pitch")
    assert_lse_close(l, rl, "padded pitch")


def test_bad_block_id_is_masked_and_flagged(m):
    case = synth.paged_case(602, synth.BF16, B=2, q_len=1, H=16, L_lo=200, L_hi=300, block_size=64)
    m.read_device_errors()
    case.block_table = case.block_table.copy()
    case.block_table[0, 1] = case.cache.shape[0] + 3
    o, l = m.paged_decode(gpu_q(case), t_u8(case.cache), t_i32(case.block_table), t_i32(case.seq_lens),
                          fmt=synth.BF16, max_context=case.max_context, softmax_scale=case.softmax_scale)
    assert m.read_device_errors() & 2


def test_config1_epilogue_then_decode_full(m):
    case, epi = synth.config1()
    cache = case.cache.copy()
    ref_q = oracle.q_concat_cache_insert(synth.BF16, epi.ql_nope, epi.q_pe, epi.kv_c, epi.k_pe, cache,
                                         epi.slot_mapping, positions=epi.positions, cos_sin=epi.cos_sin)
    gcache = t_u8(case.cache)
    gq = m.q_concat_cache_insert(t_bf16(epi.ql_nope), t_bf16(epi.q_pe), t_bf16(epi.kv_c), t_bf16(epi.k_pe), gcache,
                                 t_i64(epi.slot_mapping), fmt=synth.BF16, positions=t_i64(epi.positions),
                                 cos_sin_cache=torch.from_numpy(epi.cos_sin).cuda())
    o, l = m.paged_decode(gq, gcache, t_i32(case.block_table), t_i32(case.seq_lens), fmt=synth.BF16,
                          max_context=case.max_context, softmax_scale=case.softmax_scale, return_lse=True)
    ro, rl = oracle.paged_decode(synth.BF16, ref_q.view(np.uint8).reshape(32, 16, 1152), cache, case.block_table,
                                 case.seq_lens, 1, case.softmax_scale)
    assert np.array_equal(bf16_bits(gq), ref_q)
    assert_attn_close(o, ro, "config1")
    assert_lse_close(l, rl, "config1")
    assert m.read_device_errors() == 0


@pytest.mark.slow
def test_config3_fp8_spec_verify_all_rows(m):
    """fp8 spec-verify at full size: all 256 query rows (64 requests x 4 causal tokens) x 16
    heads, split-K over max_context 131072 and the merge."""
    case = synth.config3()
    o, l, ro, rl = run(m, case)
    assert o.shape[0] == 256
    assert_attn_close(o, ro, "config3")
    assert_lse_close(l, rl, "config3")
    assert m.read_device_errors() == 0


@pytest.mark.slow
def test_config4_ds_mla_h96_all_rows(m):
    """fp8_ds_mla decode at full size: all 128 requests x 96 heads."""
    case = synth.config4()
    o, l, ro, rl = run(m, case)
    assert l is None and o.shape[0] == 128
    assert_attn_close(o, ro, "config4")
    assert m.read_device_errors() == 0


def test_gather_dequant_bit_exact(m):
    for fmt in FMTS:
        case = synth.paged_case(700 + fmt, fmt, B=2, q_len=1, H=1, L_lo=100, L_hi=200, block_size=16)
        nslots = case.cache.shape[0] * 16
        slots = np.concatenate([np.arange(0, nslots, 7), [-1, nslots + 100]]).astype(np.int64)
        g = m.gather_dequant(t_u8(case.cache), t_i64(slots), fmt=fmt).cpu().numpy()
        flat = case.cache.reshape(-1, case.cache.shape[2])
        for i, s in enumerate(slots):
            ref = np.zeros(576) if (s < 0 or s >= nslots) else oracle.decode_entry(fmt, flat[s])
            assert np.array_equal(g[i], ref.astype(np.float32)), (fmt, s)
        assert m.read_device_errors() == 2
