"""A bounded in-kernel wait that runs out: the page kernel's consumers wait for data that the
test aid mla_debug_stall_next_decode keeps the producer from loading.  The call returns, the
device error word carries MLA_DEVERR_TIMEOUT, and the next normal call on the same context is
correct.  Nothing faults or hangs: the producer issues no copy, so none is in flight when the
consumers give up, and every role leaves through the kernel's normal teardown."""
import numpy as np
import pytest

import oracle
from mla_latent_cache_attention_gb300 import synth
from tests.gpu_helpers import assert_attn_close, assert_lse_close, t_bf16, t_i32, t_u8

pytestmark = pytest.mark.gpu
MLA_DEVERR_TIMEOUT = 16


@pytest.fixture(scope="module")
def m():
    import mla_latent_cache_attention_gb300 as mod
    mod.lib()
    return mod


def decode(m, case):
    q = t_bf16(case.q.view(np.uint16))
    return m.paged_decode(q, t_u8(case.cache), t_i32(case.block_table), t_i32(case.seq_lens), fmt=case.fmt,
                          max_context=case.max_context, softmax_scale=case.softmax_scale, return_lse=True)


def test_wait_runs_out_then_next_call_is_correct(m):
    import torch
    case = synth.paged_case(910, synth.BF16, B=3, q_len=1, H=16, L_lo=200, L_hi=400, block_size=64)
    assert m.paged_decode_workspace_size(3, 1, 16, case.max_context) == 0     # one split: no merge
    m.read_device_errors()
    m.debug_stall_next_decode(2000)           # 2 ms wait limit for that launch
    decode(m, case)
    torch.cuda.synchronize()
    assert m.read_device_errors() & MLA_DEVERR_TIMEOUT
    o, l = decode(m, case)
    ro, rl = oracle.paged_decode(case.fmt, case.q, case.cache, case.block_table, case.seq_lens, 1,
                                 case.softmax_scale)
    assert_attn_close(o, ro, "after timeout")
    assert_lse_close(l, rl, "after timeout")
    assert m.read_device_errors() == 0
