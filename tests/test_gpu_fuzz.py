"""Seeded random shapes against the fp64 oracle: the paged decode over all three cache
formats (head counts 1..128, q_len 1..5, block sizes 1..256, zero-length and short requests,
split-K from a max_context above the lengths, padded entry pitch, fp8 scales), the sparse
forward on both kernel designs (head counts 1..128, ragged and empty rows, masked and
duplicate indices) and the decode epilogue (bit-exact).  Each case is sized so that the
oracle finishes in well under a second."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import assert_attn_close, assert_lse_close, t_bf16, t_i32, t_u8

pytestmark = pytest.mark.gpu

WORK_CAP = 4e8       # oracle multiply-adds per case (rows x heads x keys x 1088)


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def paged_params(seed):
    rng = np.random.default_rng(10_000 + seed)
    fmt = int(rng.integers(0, 3))
    H = int(rng.choice([1, 2, 3, 7, 16, 20, 32, 48, 64, 96, 128]))
    q_len = int(rng.integers(1, 6))
    B = int(rng.integers(1, 7))
    bs = int(rng.choice([1, 16, 32, 64, 128, 256]))
    # lengths up to 3000, scaled down so that the oracle's work stays under the cap
    hi = int(min(3000, WORK_CAP / (B * q_len * H * 1088)))
    lens = rng.integers(0, max(hi, 2), size=B)
    short = rng.random(B) < 0.2
    lens[short] = rng.integers(0, 4, size=int(short.sum()))
    mc_mul = int(rng.choice([1, 4, 16]))
    pad = int(rng.choice([0, 0, 16, 48]))
    qs, ks = (float(rng.uniform(0.02, 0.2)), float(rng.uniform(0.02, 0.2))) if fmt == synth.FP8 else (1.0, 1.0)
    return dict(fmt=fmt, H=H, q_len=q_len, B=B, bs=bs, lens=[int(x) for x in lens], mc_mul=mc_mul, pad=pad,
                q_scale=qs, k_scale=ks)


@pytest.mark.parametrize("seed", range(80))
def test_paged_random_shapes(m, seed):
    a = paged_params(seed)
    mc = max(max(a["lens"]), 1) * a["mc_mul"]
    case = synth.paged_case(20_000 + seed, a["fmt"], B=a["B"], q_len=a["q_len"], H=a["H"], L_lo=0, L_hi=3000,
                            block_size=a["bs"], max_context=mc, entry_pad=a["pad"], q_scale=a["q_scale"],
                            k_scale=a["k_scale"], seq_lens=a["lens"])
    q = t_u8(case.q) if case.fmt == synth.FP8 else t_bf16(case.q.view(np.uint16))
    m.read_device_errors()
    o, l = m.paged_decode(q, t_u8(case.cache), t_i32(case.block_table), t_i32(case.seq_lens), fmt=case.fmt,
                          q_len=case.q_len, max_context=mc, softmax_scale=case.softmax_scale, q_scale=case.q_scale,
                          k_scale=case.k_scale, return_lse=True)
    ro, rl = oracle.paged_decode(case.fmt, case.q, case.cache, case.block_table, case.seq_lens, case.q_len,
                                 case.softmax_scale, case.q_scale, case.k_scale)
    assert_attn_close(o, ro, f"paged {a}")
    assert_lse_close(l, rl, f"paged {a}")
    assert m.read_device_errors() == 0


def sparse_params(seed):
    rng = np.random.default_rng(30_000 + seed)
    T = int(rng.integers(1, 41))
    H = int(rng.choice([1, 3, 8, 16, 17, 31, 32, 64, 100, 128]))
    N = int(rng.integers(1, 3000))
    per_row = int(rng.integers(0, max(2, int(min(700, WORK_CAP / (T * H * 1088))))))
    return dict(T=T, H=H, N=N, per_row=per_row, p_invalid=float(rng.choice([0.0, 0.1, 0.5])),
                replace=bool(rng.integers(0, 2)) or per_row > N, ragged=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("kern", ["gather", "staged"])
@pytest.mark.parametrize("seed", range(40))
def test_sparse_random_shapes(m, seed, kern):
    a = sparse_params(seed)
    c = synth.sparse_case(40_000 + seed, **a)
    m.read_device_errors()
    o, l = m.sparse_fwd(t_bf16(c.q), t_u8(c.records), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=c.has_invalid, return_lse=True, kernel=kern)
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, c.has_invalid)
    assert_attn_close(o, ro, f"sparse {a}")
    assert_lse_close(l, rl, f"sparse {a}")
    assert m.read_device_errors() == 0


@pytest.mark.parametrize("seed", range(40))
def test_epilogue_random_shapes(m, seed):
    """The decode epilogue (q concat + latent insert), bit-exact: random format, batch, head
    count, block size, pitch, RoPE on / off and skipped slots."""
    from tests.test_gpu_epilogue import run_both
    rng = np.random.default_rng(50_000 + seed)
    fmt = int(rng.integers(0, 3))
    B = int(rng.integers(1, 65))
    H = int(rng.choice([1, 2, 5, 16, 33, 64, 128]))
    bs = int(rng.choice([1, 4, 16, 64]))
    nb = int(np.ceil(B / bs)) + int(rng.integers(0, 5))
    run_both(m, fmt, B=B, H=H, bs=bs, nb=nb, seed=60_000 + seed, rope=bool(rng.integers(0, 2)),
             entry_pad=int(rng.choice([0, 16, 48])), neg_slot=bool(rng.integers(0, 2)))
