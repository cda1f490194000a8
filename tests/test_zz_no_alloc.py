"""mla_paged_decode_noalloc: the paged decode for callers that cannot allocate device memory
(code running where cudaMalloc is not allowed, plug-ins whose host engine owns all device
memory, serving loops that forbid allocation).  It keeps its split-K partials in a static
scratch array inside the library.

Called through the C ABI, its output must match mla_paged_decode (caller workspace) within
the attention tolerance, on two calls in a row (the second sees the first call's scratch
contents).  This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import ATOL, LSE_TOL, RTOL, t_bf16, t_i32, t_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from mla_latent_cache_attention_gb300 import build
    build.build()
    import mla_latent_cache_attention_gb300 as m
    return m.lib()


def _decode_both(L, case):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q = t_u8(case.q) if case.fmt == synth.FP8 else t_bf16(case.q.view(np.uint16))
    cache, bt, sl = t_u8(case.cache), t_i32(case.block_table), t_i32(case.seq_lens)
    B, rows, H = case.seq_lens.size, case.q.shape[0], case.H
    nb, bs, es = case.cache.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    outs = []
    for noalloc in (False, True):
        out = torch.full((rows, H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((rows, H), float("nan"), dtype=torch.float32, device=dev)
        common = [ctypes.c_void_p(q.data_ptr()), q.stride(0), q.stride(1), ctypes.c_void_p(cache.data_ptr()),
                  case.fmt, nb, bs * es, es, bs, ctypes.c_void_p(bt.data_ptr()), bt.stride(0),
                  ctypes.c_void_p(sl.data_ptr()), B, case.q_len, H, case.max_context, case.softmax_scale,
                  case.q_scale, case.k_scale, ctypes.c_void_p(out.data_ptr()), out.stride(0), out.stride(1),
                  ctypes.c_void_p(lse.data_ptr())]
        if noalloc:
            rc = L.mla_paged_decode_noalloc(*common, stream)
        else:
            need = L.mla_paged_decode_workspace_size(B, case.q_len, H, case.max_context, 0)
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            rc = L.mla_paged_decode(*common, ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream)
        assert rc == 0, L.mla_last_error()
        torch.cuda.synchronize()
        outs.append((out.float().cpu().numpy(), lse.cpu().numpy()))
    return outs


@pytest.mark.parametrize("fmt", [synth.BF16, synth.DS_MLA])
def test_noalloc_matches_workspace_version_twice(L, fmt):
    # the split count is high enough that the partials go through the scratch
    assert L.mla_paged_decode_workspace_size(4, 2, 16, 32768, 0) > 0
    for call, seed in enumerate((11, 12)):
        case = synth.paged_case(seed + 10 * fmt, fmt, B=4, q_len=2, H=16, L_lo=500 + 900 * call, L_hi=9000,
                                block_size=64, max_context=32768)
        (o_ref, l_ref), (o_na, l_na) = _decode_both(L, case)
        assert np.all(np.isfinite(o_na))
        assert np.all(np.abs(o_na - o_ref) <= ATOL + RTOL * np.abs(o_ref)), f"call {call}"
        fin = np.isfinite(l_ref)
        assert np.array_equal(fin, np.isfinite(l_na))
        assert np.all(np.abs(l_na[fin] - l_ref[fin]) <= LSE_TOL), f"call {call}"


def test_noalloc_rejects_shapes_beyond_its_scratch(L):
    # find a batch whose split-K partials need more than the 64 MiB static scratch
    big = next(b for b in range(16, 4096, 8) if L.mla_paged_decode_workspace_size(b, 1, 16, 1 << 16, 0) > (64 << 20))
    fake = ctypes.c_void_p(1 << 20)
    rc = L.mla_paged_decode_noalloc(fake, 16 * 576, 576, fake, 0, 10, 64 * 1152, 1152, 64, fake, 1024, fake,
                                    big, 1, 16, 1 << 16, 0.1, 1.0, 1.0, fake, 16 * 512, 512, None, None)
    assert rc == -2
    assert b"static scratch holds" in L.mla_last_error()
