"""fp8_ds_mla paged decode run by clusters of 2, 3 or 6 CTAs (sharing each page tile through
multicast copies) against one CTA per head group: the same bits, and both against the fp64
oracle.  Shapes cover one and several clusters per request, spec-verify columns, split-K
with empty splits, zero-length requests, block sizes below and above the 128-key tile, a
group count that no cluster size divides (served one CTA per group) and a bad block id."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import assert_attn_close, assert_lse_close, t_bf16, t_i32, t_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    yield mod
    mod.debug_ds_cluster(0)


def runs(m, case, sizes, max_context=None, bt=None):
    mc = case.max_context if max_context is None else max_context
    q = t_bf16(case.q.view(np.uint16))
    cache, sl = t_u8(case.cache), t_i32(case.seq_lens)
    bt = t_i32(case.block_table if bt is None else bt)
    res = []
    for size in sizes:
        m.debug_ds_cluster(size)
        res.append(m.paged_decode(q, cache, bt, sl, fmt=case.fmt, q_len=case.q_len, max_context=mc,
                                  softmax_scale=case.softmax_scale, return_lse=True))
    m.debug_ds_cluster(0)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("H,q_len,bs,mc", [(32, 1, 64, None), (96, 1, 64, 65536), (16, 2, 64, None),
                                           (128, 1, 16, None), (64, 1, 256, 65536), (48, 1, 64, None),
                                           (96, 2, 32, 32768)])
def test_clusters_match_single_ctas_and_oracle(m, H, q_len, bs, mc):
    lens = [0, 1, 129, 700, 2500, 255, 1024, 3000]
    case = synth.paged_case(900 + H + q_len + bs, synth.DS_MLA, B=len(lens), q_len=q_len, H=H, L_lo=1, L_hi=3000,
                            block_size=bs, seq_lens=lens)
    m.read_device_errors()
    res = runs(m, case, [1, 2, 3, 6, 0], max_context=mc)
    os_, ls = res[0]
    for size, (o, l) in zip([2, 3, 6, 0], res[1:]):
        assert torch.equal(o, os_), f"cluster size {size} and single CTAs differ"
        assert torch.equal(l, ls)
    op, lp = res[-1]
    assert m.read_device_errors() == 0
    ro, rl = oracle.paged_decode(case.fmt, case.q, case.cache, case.block_table, case.seq_lens, case.q_len,
                                 case.softmax_scale, 1.0, 1.0)
    assert_attn_close(op, ro, f"pairs H={H} q={q_len} bs={bs}")
    assert_lse_close(lp, rl, f"pairs H={H} q={q_len} bs={bs}")


def test_clusters_bad_block_id_is_masked_and_flagged(m):
    case = synth.paged_case(977, synth.DS_MLA, B=3, q_len=1, H=96, L_lo=300, L_hi=600, block_size=64)
    bt = case.block_table.copy()
    bt[1, 2] = case.cache.shape[0] + 5
    for size in (2, 3, 6):
        m.read_device_errors()
        (o1, l1), (oc, lc) = runs(m, case, [1, size], bt=bt)
        assert m.read_device_errors() & 2
        assert torch.equal(o1, oc) and torch.equal(l1, lc)
