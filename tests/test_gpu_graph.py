"""The entry points are safe to capture in a CUDA graph (no host synchronisation, no
allocation by the library, tensor maps passed by value): a captured step replays to the same
bits as direct calls -- the decode epilogue + paged decode with split-K and the merge
(programmatic dependent launch inside the graph), and the sparse forward."""
import numpy as np
import pytest
import torch

from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import t_bf16, t_i32, t_i64, t_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                    # first call (tensor maps, device info) outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_step_graph_replays_bit_exact(m):
    case, epi = synth.config1(B=8, L_lo=2000, L_hi=8000)
    cache0 = t_u8(case.cache)
    cache = cache0.clone()
    ws = torch.empty(max(m.paged_decode_workspace_size(8, 1, 16, 65536), 256), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 256                                   # split-K: the merge runs too
    mqa = torch.empty((8, 16, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((8, 16, 512), dtype=torch.bfloat16, device="cuda")
    args = [t_bf16(epi.ql_nope), t_bf16(epi.q_pe), t_bf16(epi.kv_c), t_bf16(epi.k_pe)]
    slots, pos, cs = t_i64(epi.slot_mapping), t_i64(epi.positions), torch.from_numpy(epi.cos_sin).cuda()
    bt, sl = t_i32(case.block_table), t_i32(case.seq_lens)

    def step():
        q = m.q_concat_cache_insert(*args, cache, slots, fmt=synth.BF16, positions=pos, cos_sin_cache=cs, mqa_q=mqa)
        m.paged_decode(q, cache, bt, sl, fmt=synth.BF16, max_context=65536, softmax_scale=case.softmax_scale,
                       out=out, workspace=ws)

    step()
    torch.cuda.synchronize()
    ref_out, ref_cache = out.clone(), cache.clone()
    out.zero_()
    cache.copy_(cache0)
    g = capture(step)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(cache, ref_cache)
    assert m.read_device_errors() == 0


def test_sparse_graph_replays_bit_exact(m):
    c = synth.config2(T=128)
    q, rec, ptr, idx = t_bf16(c.q), t_u8(c.records), t_i32(c.indptr), t_i32(c.indices)
    out = torch.empty((128, 16, 512), dtype=torch.bfloat16, device="cuda")
    res = {}

    def step():
        res["lse"] = m.sparse_fwd(q, rec, ptr, idx, c.softmax_scale, has_invalid=True, out=out, return_lse=True)[1]

    step()
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), res["lse"].clone()
    g = capture(step)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(res["lse"], ref_lse)


def test_ds_cluster_decode_graph_replays_bit_exact(m):
    """The fp8_ds_mla decode of 96 heads runs as 2-CTA clusters (multicast page tiles), with
    split-K and the merge: captured and replayed, it gives the direct call's bits."""
    case = synth.paged_case(61, synth.DS_MLA, B=6, q_len=1, H=96, L_lo=1500, L_hi=5000, block_size=64,
                            max_context=32768)
    q, cache = t_bf16(case.q.view(np.uint16)), t_u8(case.cache)
    bt, sl = t_i32(case.block_table), t_i32(case.seq_lens)
    ws = torch.empty(max(m.paged_decode_workspace_size(6, 1, 96, 32768), 256), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 256
    out = torch.empty((6, 96, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((6, 96), dtype=torch.float32, device="cuda")

    def step():
        m.paged_decode(q, cache, bt, sl, fmt=synth.DS_MLA, max_context=32768, softmax_scale=case.softmax_scale,
                       out=out, workspace=ws, lse=lse)

    step()
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    g = capture(step)
    for _ in range(3):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    assert m.read_device_errors() == 0
