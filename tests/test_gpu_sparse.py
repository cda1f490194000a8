"""GPU parity of the sparse forward (CSR over fp8_ds_mla records) against the fp64 oracle:
the tiny configuration in full, edge cases (empty / all-masked / ragged rows, duplicates,
head counts that are not multiples of 16, strided out, no lse), and the full-size prefill
configuration on sampled rows."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import assert_attn_close, assert_lse_close, t_bf16, t_i32, t_u8

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def run(m, c: synth.SparseCase, rows=None, out=None, lse=True):
    q = t_bf16(c.q)
    o, l = m.sparse_fwd(q, t_u8(c.records), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=c.has_invalid, out=out, return_lse=lse)
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, c.has_invalid, rows=rows)
    if rows is not None:
        o = o[torch.as_tensor(rows, device=o.device)]
        l = l[torch.as_tensor(rows, device=o.device)] if l is not None else None
    return o, l, ro, rl


def test_config0_tiny(m):
    c = synth.config0()
    o, l, ro, rl = run(m, c)
    assert_attn_close(o, ro, "config0 out")
    assert_lse_close(l, rl, "config0 lse")
    assert torch.all(o[3] == 0) and torch.all(l[3] == -np.inf)
    assert m.read_device_errors() == 0


def test_golden_warmup_problem(m):
    g = json.load(open(os.path.join(GOLDEN, "warmup_one_token.json")))
    rec = torch.zeros((1, 656), dtype=torch.uint8, device="cuda")
    for H in g["heads"]:
        q = torch.zeros((1, H, 576), dtype=torch.bfloat16, device="cuda")
        o, l = m.sparse_fwd(q, rec, t_i32(g["indptr"]), t_i32(g["indices"]), g["softmax_scale"], return_lse=True)
        assert torch.all(o == g["expected_out"]) and torch.all(l == g["expected_lse"])


@pytest.mark.parametrize("H", [1, 5, 16, 20, 64, 96, 128])
def test_head_counts(m, H):
    c = synth.sparse_case(100 + H, T=6, H=H, N=500, per_row=200, p_invalid=0.1, replace=True, ragged=True)
    o, l, ro, rl = run(m, c)
    assert_attn_close(o, ro, f"H={H}")
    assert_lse_close(l, rl, f"H={H}")


def test_multi_tile_ragged_rows(m):
    # row lengths 0, 1, 127, 128, 129, 255, 256, 257, 1000, all-masked
    lens = [0, 1, 127, 128, 129, 255, 256, 257, 1000, 40]
    rng = np.random.default_rng(5)
    c = synth.sparse_case(5, T=len(lens), H=16, N=3000, per_row=1, p_invalid=0.0, replace=True)
    ptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = rng.integers(0, 3000, size=ptr[-1]).astype(np.int32)
    idx[rng.random(idx.size) < 0.07] = -1
    idx[ptr[-2]:ptr[-1]] = -1                    # last row fully masked
    c.q = synth.normal_bf16_bits(rng, (len(lens), 16, 576))
    c.indptr, c.indices, c.has_invalid = ptr, idx, True
    o, l, ro, rl = run(m, c)
    assert_attn_close(o, ro, "ragged")
    assert_lse_close(l, rl, "ragged")
    assert torch.all(o[0] == 0) and torch.all(o[-1] == 0)


def test_duplicates_without_has_invalid_and_no_lse(m):
    c = synth.sparse_case(9, T=8, H=16, N=50, per_row=300, p_invalid=0.0, replace=True)
    o, l, ro, rl = run(m, c, lse=False)
    assert l is None
    assert_attn_close(o, ro, "duplicates")


def test_strided_out_and_q(m):
    c = synth.sparse_case(13, T=5, H=16, N=400, per_row=150, p_invalid=0.05, replace=False)
    qbig = torch.zeros((5, 16, 640), dtype=torch.bfloat16, device="cuda")
    qbig[:, :, :576] = t_bf16(c.q)
    out = torch.full((5, 16, 600), 7.0, dtype=torch.bfloat16, device="cuda")
    o, l = m.sparse_fwd(qbig[:, :, :576], t_u8(c.records), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=True, out=out[:, :, :512], return_lse=True)
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True)
    assert_attn_close(out[:, :, :512], ro, "strided")
    assert torch.all(out[:, :, 512:] == 7.0)
    assert_lse_close(l, rl, "strided")


def test_padded_record_pitch(m):
    c = synth.sparse_case(17, T=4, H=16, N=300, per_row=200, p_invalid=0.1, replace=True)
    padded = np.zeros((300, 672), dtype=np.uint8)
    padded[:, :656] = c.records
    o, l = m.sparse_fwd(t_bf16(c.q), t_u8(padded), t_i32(c.indptr), t_i32(c.indices), c.softmax_scale,
                        has_invalid=True, return_lse=True)
    ro, rl = oracle.sparse_fwd(c.q, padded, c.indptr, c.indices, c.softmax_scale, True)
    assert_attn_close(o, ro, "padded pitch")
    assert_lse_close(l, rl, "padded pitch")


def test_power_of_two_and_large_scales(m):
    rng = np.random.default_rng(21)
    c = synth.sparse_case(21, T=4, H=16, N=256, per_row=256, p_invalid=0.0, replace=False)
    c.records[:, 512:528] = (2.0 ** rng.integers(-6, 8, size=(256, 4))).astype(np.float32).view(np.uint8)
    o, l, ro, rl = run(m, c)
    assert_attn_close(o, ro, "pow2 scales")
    # scales up to 2^7 put |lse| near 3e4, where fp32 resolution is 2e-3: allow 1e-6 relative
    assert_lse_close(l, rl, "pow2 scales", rel=1e-6)


def test_out_of_range_index_is_masked_and_flagged(m):
    c = synth.sparse_case(23, T=3, H=16, N=100, per_row=50, p_invalid=0.0, replace=True)
    m.read_device_errors()
    bad = c.indices.copy()
    bad[7] = 100
    q = t_bf16(c.q)
    o, l = m.sparse_fwd(q, t_u8(c.records), t_i32(c.indptr), t_i32(bad), c.softmax_scale, return_lse=True)
    assert m.read_device_errors() & 1
    masked = bad.copy()
    masked[7] = -1
    ro, rl = oracle.sparse_fwd(c.q, c.records, c.indptr, masked, c.softmax_scale, True)
    assert_attn_close(o, ro, "masked bad index")


@pytest.mark.slow
def test_config2_full_size_sampled_rows(m):
    c = synth.config2()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, c.q.shape[0] - 1], rng.choice(c.q.shape[0], 61, replace=False)]))
    o, l, ro, rl = run(m, c, rows=rows)
    assert_attn_close(o, ro, "config2")
    assert_lse_close(l, rl, "config2")
    assert m.read_device_errors() == 0


def test_staged_converter_variant():
    # the staged-converter kernel (selected per process by MLA_SPARSE_GATHER=0) against the
    # same cases, full-size prefill included, in a child process
    import subprocess
    import sys
    env = dict(os.environ, MLA_SPARSE_GATHER="0")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.abspath(__file__), "-m", "gpu", "-q", "-x",
                        "-p", "no:cacheprovider", "-k", "not staged_converter_variant"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
