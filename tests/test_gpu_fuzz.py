"""Seeded random shapes against the fp64 oracle: the paged decode over all three cache
formats (head counts 1..128, q_len 1..5, block sizes 1..256, zero-length and short requests,
split-K from a max_context above the lengths, padded entry pitch, fp8 scales), the sparse
forward on both kernel designs (head counts 1..128, ragged and empty rows, masked and
duplicate indices), the decode and prefill epilogues and the chunked-context gather
(bit-exact), the prefix / suffix merge and the absorbed per-head contractions.  Each case is
sized so that the oracle finishes in well under a second."""
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


@pytest.mark.parametrize("seed", range(200))
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


def test_paged_ds_cancellation_case(m):
    """A random ds_mla shape (H=128, q_len=3, block 128, a 14-key request) whose output -0.06
    cancels values near 448 times a 0.1 scale: with P_j carried only as its f16 value it fell
    1.1 times outside the tolerance; the fp32-rounded first P term keeps it inside."""
    test_paged_random_shapes(m, 20233)


def sparse_params(seed):
    rng = np.random.default_rng(30_000 + seed)
    T = int(rng.integers(1, 41))
    H = int(rng.choice([1, 3, 8, 16, 17, 31, 32, 64, 100, 128]))
    N = int(rng.integers(1, 3000))
    per_row = int(rng.integers(0, max(2, int(min(700, WORK_CAP / (T * H * 1088))))))
    return dict(T=T, H=H, N=N, per_row=per_row, p_invalid=float(rng.choice([0.0, 0.1, 0.5])),
                replace=bool(rng.integers(0, 2)) or per_row > N, ragged=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("kern", ["gather", "staged"])
@pytest.mark.parametrize("seed", range(100))
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


@pytest.mark.parametrize("seed", range(20))
def test_prefill_epilogues_random_shapes(m, seed):
    """The prefill epilogues, bit-exact: key concat + latent insert (bf16 / fp8_ds_mla) and the
    fp8 q / k / v quantisation + insert, over random token counts, heads, block sizes,
    pitches, skipped slots and RoPE on / off."""
    from tests.gpu_helpers import bf16_bits, t_i64
    from tests.test_gpu_prefill_epilogue import dev_rope, inputs
    rng = np.random.default_rng(70_000 + seed)
    Tp = int(rng.integers(1, 48))
    H = int(rng.choice([1, 3, 8, 16, 20, 33]))
    bs = int(rng.choice([1, 8, 16, 64]))
    nb = int(np.ceil(Tp / bs)) + int(rng.integers(0, 4))
    rope = bool(rng.integers(0, 2))
    skip = tuple(int(t) for t in rng.choice(Tp, size=min(Tp, int(rng.integers(0, 3))), replace=False))
    pad = int(rng.choice([0, 16]))
    fmt = int(rng.choice([synth.BF16, synth.DS_MLA, synth.FP8]))
    d, cache = inputs(71_000 + seed, Tp=Tp, H=H, nb=nb, bs=bs, fmt=fmt, rope=rope, skip=skip, entry_pad=pad)
    ref_cache = cache.copy()
    gcache = t_u8(cache)
    pos, cs = dev_rope(d)
    m.read_device_errors()
    if fmt != synth.FP8:
        ref_q = d["q"].copy()
        ref_k = oracle.key_concat_cache_insert(fmt, ref_q, d["k_nope"], d["k_pe"], d["kv_c"], ref_cache, d["slots"],
                                               positions=d["pos"], cos_sin=d["cs"])
        q = t_bf16(d["q"])
        k_out = m.key_concat_cache_insert(q, t_bf16(d["k_nope"]), t_bf16(d["k_pe"]), t_bf16(d["kv_c"]), gcache,
                                          t_i64(d["slots"]), fmt=fmt, positions=pos, cos_sin_cache=cs)
        assert np.array_equal(bf16_bits(k_out), ref_k)
        assert np.array_equal(bf16_bits(q), ref_q)
    else:
        sc = {k: float(np.float32(v)) for k, v in dict(q_scale_inv=1 / 0.05, k_scale_inv=1 / 0.03,
                                                         v_scale_inv=1 / 0.02, cache_scale_inv=1 / 0.07).items()}
        rq, rk, rv = oracle.qkv_quant_cache_fp8_insert(d["q"], d["k_nope"], d["k_pe"], d["kv_c"], d["v"], ref_cache,
                                                       d["slots"], positions=d["pos"], cos_sin=d["cs"], **sc)
        dsc = {k: torch.tensor([v], dtype=torch.float32, device="cuda") for k, v in sc.items()}
        q8, k8, v8 = m.qkv_quant_cache_fp8_insert(t_bf16(d["q"]), t_bf16(d["k_nope"]), t_bf16(d["k_pe"]),
                                                  t_bf16(d["kv_c"]), t_bf16(d["v"]), gcache, t_i64(d["slots"]),
                                                  positions=pos, cos_sin_cache=cs, **dsc)
        assert np.array_equal(q8.cpu().numpy(), rq)
        assert np.array_equal(k8.cpu().numpy(), rk)
        assert np.array_equal(v8.cpu().numpy(), rv)
    assert np.array_equal(gcache.cpu().numpy(), ref_cache)
    assert m.read_device_errors() == 0


@pytest.mark.parametrize("seed", range(20))
def test_chunked_context_random_shapes(m, seed):
    """The chunked-context gather (bit-exact, up-converted or raw) and the prefix / suffix
    merge, over random formats, block sizes, chunk layouts, head counts, head dims and empty
    sides."""
    from tests.gpu_helpers import bf16_bits
    from tests.test_gpu_chunked_context import check_merge, chunk_of, merge_inputs
    rng = np.random.default_rng(80_000 + seed)
    fmt = int(rng.integers(0, 3))
    raw = bool(rng.integers(0, 2))
    bs = int(rng.choice([1, 16, 64, 128]))
    B = int(rng.integers(2, 8))
    case = synth.paged_case(81_000 + seed, fmt, B=B, q_len=1, H=1, L_lo=1, L_hi=800, block_size=bs,
                            entry_pad=int(rng.choice([0, 16])), q_scale=0.05, k_scale=float(rng.uniform(0.02, 0.1)))
    cu, starts = chunk_of(case, rng)
    n = int(cu[-1]) + int(rng.integers(0, 4))
    ref = oracle.gather_context(fmt, case.cache, case.block_table, cu, starts, num_tokens=n, raw=raw,
                                scale=case.k_scale)
    dst = m.gather_context(t_u8(case.cache), t_i32(case.block_table), t_i32(cu), t_i32(starts), fmt=fmt,
                           num_tokens=n, raw=raw, scale=case.k_scale)
    got = dst.cpu().numpy() if raw else bf16_bits(dst)
    assert np.array_equal(got[:cu[-1]], ref[:cu[-1]])
    T, H, D = int(rng.integers(1, 50)), int(rng.choice([1, 4, 16, 20])), int(rng.choice([64, 100, 128, 512]))
    pick = lambda: tuple(int(t) for t in rng.choice(T, size=min(T, int(rng.integers(0, 3))), replace=False))
    a, lp, b, ls = merge_inputs(82_000 + seed, T, H, D, empty_p=pick(), empty_s=pick(), both=pick())
    ref, rl = oracle.merge_attn_states(a, lp, b, ls)
    out, lse = m.merge_attn_states(t_bf16(a), torch.from_numpy(lp).cuda(), t_bf16(b), torch.from_numpy(ls).cuda(),
                                   return_lse=True)
    check_merge(out, lse, ref, rl, a, b)
    assert m.read_device_errors() == 0


@pytest.mark.parametrize("seed", range(16))
def test_absorbed_contractions_random_shapes(m, seed):
    """The absorbed decode's per-head contractions on the tensor cores (BMM1 with W_UK_T, W_UV
    with and without the sigmoid gate) over random batches, head counts and inner sizes,
    within one bf16 rounding per step plus fp32 accumulation of the fp64 product."""
    from tests.gpu_helpers import bf16_bits
    from tests.test_gpu_absorb import check, weights
    rng = np.random.default_rng(90_000 + seed)
    B = int(rng.integers(1, 150))
    H = int(rng.choice([1, 2, 16, 24, 96, 128]))
    P = int(rng.choice([64, 128, 192, 512]))
    q = synth.normal_bf16_bits(rng, (B, H, P))
    w = weights(rng, H, P, 512)
    ql = m.absorb_q(t_bf16(q), t_bf16(w))
    check(bf16_bits(ql), q, w, oracle.head_bmm(q, w))
    V = int(rng.choice([128, 256]))
    lat = synth.normal_bf16_bits(rng, (B, H, 512))
    wv = weights(rng, H, 512, V)
    gated = bool(rng.integers(0, 2))
    g = synth.normal_bf16_bits(rng, (B, H * V)) if gated else None
    out = m.v_up_proj(t_bf16(lat), t_bf16(wv), None if g is None else t_bf16(g))
    check(bf16_bits(out), lat, wv, oracle.head_bmm(lat, wv, g), gate_terms=3 if gated else 1)


@pytest.mark.parametrize("seed", range(20))
def test_sparse_extras_random_shapes(m, seed):
    """The sparse forward's extras (per-head sink, second key segment, kv_splits) in random
    combinations over random row lengths, head counts and masks."""
    from tests.test_gpu_sparse_ext import run, second_segment
    rng = np.random.default_rng(95_000 + seed)
    T = int(rng.integers(1, 24))
    H = int(rng.choice([1, 5, 16, 20, 64, 128]))
    hi = int(max(2, min(1500, WORK_CAP / (T * H * 1088 * 2))))
    lens = rng.integers(0, hi, size=T)
    N = int(rng.integers(1, 2500))
    c = synth.sparse_case(96_000 + seed, T=T, H=H, N=N, per_row=1, p_invalid=0.0, replace=True)
    c.indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    c.indices = rng.integers(0, N, size=c.indptr[-1]).astype(np.int32)
    c.indices[rng.random(c.indices.size) < float(rng.choice([0.0, 0.1, 0.6]))] = -1
    c.q = synth.normal_bf16_bits(rng, (T, H, 576))
    sink = None
    if rng.integers(0, 2):
        sink = rng.uniform(-5.0, 20.0, size=H).astype(np.float32)
        sink[rng.random(H) < 0.2] = -np.inf
    seg = second_segment(97_000 + seed, T, N2=int(rng.integers(1, 800)), hi=hi) if rng.integers(0, 2) else None
    kv_splits = int(rng.choice([1, 1, 2, 3, 7]))
    if sink is None and seg is None and kv_splits == 1:
        kv_splits = 2
    m.read_device_errors()
    o, l, ro, rl = run(m, c, sink=sink, seg=seg, kv_splits=kv_splits)
    what = f"T={T} H={H} sink={sink is not None} seg={seg is not None} kv_splits={kv_splits}"
    assert_attn_close(o, ro, what)
    assert_lse_close(l, rl, what)
    assert m.read_device_errors() == 0
