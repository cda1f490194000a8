"""The C-ABI library loads, exports every symbol include/mla.h declares, and rejects bad
arguments on the host (no GPU work: every call below fails validation or has size zero)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mla_latent_cache_attention_gb300 import build
    build.build()
    import mla_latent_cache_attention_gb300 as m
    return m.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("mla_sparse_fwd", "mla_paged_decode", "mla_q_concat_cache_insert",
              "mla_paged_decode_workspace_size", "mla_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_no_torch_types_in_the_header():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    assert "torch" not in src.replace("no torch", "") and "at::" not in src and "Tensor" not in src


def test_version_and_empty_error(L):
    assert b"sm_103a" in L.mla_version()


NULL = None


def test_sparse_rejects_bad_arguments(L):
    # H out of range -> unsupported; T == 0 -> OK without launching; NULL q -> invalid
    assert L.mla_sparse_fwd(NULL, 576, 576, NULL, 656, 1, NULL, NULL, 0, 1.0, 0, NULL, 512, 512, NULL, 4, 0, NULL) == -2
    assert b"H must be" in L.mla_last_error()
    assert L.mla_sparse_fwd(NULL, 576, 576, NULL, 656, 1, NULL, NULL, 0, 1.0, 0, NULL, 512, 512, NULL, 0, 16, NULL) == 0
    assert L.mla_sparse_fwd(NULL, 576, 576, NULL, 656, 1, NULL, NULL, 0, 1.0, 0, NULL, 512, 512, NULL, 4, 16, NULL) == -1
    fake = ctypes.c_void_p(1 << 20)
    # record pitch not a multiple of 16
    assert L.mla_sparse_fwd(fake, 576 * 16, 576, fake, 660, 10, fake, fake, 4, 1.0, 0, fake, 512 * 16, 512, NULL, 4, 16, NULL) == -1
    assert b"pitch" in L.mla_last_error()
    # index count beyond int32
    assert L.mla_sparse_fwd(fake, 576 * 16, 576, fake, 656, 10, fake, fake, 1 << 31, 1.0, 0, fake, 512 * 16, 512, NULL, 4, 16, NULL) == -2


def test_paged_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(1 << 20)
    args = lambda **kw: [kw.get("q", fake), 576 * 16, 576, fake, kw.get("fmt", 0), 10, 64 * 1152, kw.get("es", 1152), 64,
                         fake, 4, fake, kw.get("B", 2), kw.get("ql", 1), kw.get("H", 16), kw.get("mc", 4096),
                         0.1, 1.0, 1.0, fake, 512 * 16, 512, NULL, NULL, 0, NULL]
    assert L.mla_paged_decode(*args(fmt=7)) == -1
    assert L.mla_paged_decode(*args(H=129)) == -2
    assert L.mla_paged_decode(*args(B=0)) == 0
    assert L.mla_paged_decode(*args(mc=0)) == -1
    assert L.mla_paged_decode(*args(es=1000)) == -1        # entry stride below 1152
    assert L.mla_paged_decode(*args(q=NULL)) == -1


def test_epilogue_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(1 << 20)

    def call(fmt=0, qinv=NULL, cinv=NULL, pos=NULL, cs=NULL, B=2):
        return L.mla_q_concat_cache_insert(fake, 16 * 512, 512, fake, 16 * 64, 64, fake, 512, fake, 64, fake, fake,
                                           fmt, 10, 64 * 1152, 1152, 64, fake, qinv, cinv, pos, cs, 100, B, 16, NULL)
    assert call(fmt=1) == -1                    # fp8 without scales
    assert call(fmt=0, qinv=fake, cinv=fake) == -1   # scales on a bf16 cache
    assert call(pos=fake) == -1                 # positions without table
    assert call(B=0) == 0


def test_workspace_size_is_host_only_and_depends_on_the_bound_not_the_lengths(L):
    L.mla_paged_decode_workspace_size.restype = ctypes.c_size_t
    a = L.mla_paged_decode_workspace_size(64, 4, 16, 131072, 152)
    b = L.mla_paged_decode_workspace_size(64, 4, 16, 65536, 152)
    assert a > 0 and b > 0
    assert L.mla_paged_decode_workspace_size(32, 1, 16, 128, 152) == 0   # one tile: no split
    assert L.mla_paged_decode_workspace_size(0, 1, 16, 8192, 152) == 0


def test_prefill_epilogues_reject_bad_arguments(L):
    # every call below fails validation or has size zero: nothing reaches a launch
    fake = ctypes.c_void_p(1 << 20)

    def kc(fmt=0, dn=128, Tp=4, q=fake, kout=fake, pos=NULL, cs=NULL):
        return L.mla_key_concat_cache_insert(q, 16 * 192, 192, fake, 16 * 128, 128, fake, 64, fake, 512, kout, fake,
                                             fmt, 10, 64 * 1152, 1152, 64, fake, pos, cs, 100, Tp, 16, dn, NULL)
    assert kc(fmt=1) == -1                       # the plain fp8 cache has its own entry point
    assert kc(dn=100) == -2                      # NoPE head dim not a multiple of 8
    assert kc(Tp=0) == 0
    assert kc(q=NULL) == -1
    assert kc(kout=NULL) == -1
    assert kc(pos=fake) == -1                    # positions without a table

    def qkv(dv=128, Tp=4, sc=fake):
        return L.mla_qkv_quant_cache_fp8_insert(fake, 16 * 192, 192, fake, 16 * 128, 128, fake, 64, fake, 512, fake,
                                                16 * dv, dv, fake, fake, fake, fake, 10, 64 * 576, 576, 64, fake, sc,
                                                sc, sc, sc, NULL, NULL, 0, Tp, 16, 128, dv, NULL)
    assert qkv(dv=12) == -2
    assert qkv(sc=NULL) == -1
    assert qkv(Tp=0) == 0


def test_chunk_gather_and_merge_reject_bad_arguments(L):
    # every call below fails validation or has size zero: nothing reaches a launch
    fake = ctypes.c_void_p(1 << 20)

    def g(kind=0, fmt=2, row=1152, batch=2, n=10):
        return L.mla_gather_context(fake, fmt, 10, 64 * 656, 656, 64, fake, 4, fake, NULL, batch, n, kind, 1.0, fake,
                                    row, NULL)
    assert g(kind=2) == -1
    assert g(fmt=5) == -1
    assert g(row=1000) == -1                     # rows overlap for bf16 output
    assert g(batch=0) == 0 and g(n=0) == 0

    def mg(T=3, D=128, ps1=128):
        return L.mla_merge_attn_states(fake, 16 * D, D, NULL, fake, 16 * ps1, ps1, fake, fake, 16 * D, D, fake, T, 16,
                                       D, NULL)
    assert mg(T=0) == 0
    assert mg(D=0) == -1
    assert mg(ps1=64) == -1                      # prefix rows overlap


def test_sparse_ext_and_head_bmm_reject_bad_arguments(L):
    fake = ctypes.c_void_p(1 << 20)
    L.mla_sparse_fwd_ext_workspace_size.restype = ctypes.c_size_t
    assert L.mla_sparse_fwd_ext_workspace_size(4, 16, 1, 0, 0) == 0          # nothing beyond the plain forward
    assert L.mla_sparse_fwd_ext_workspace_size(4, 16, 2, 0, 0) > 0
    assert L.mla_sparse_fwd_ext_workspace_size(4, 16, 1, 0, 1) > 0           # a sink needs the partials

    def ext(splits=2, extra=NULL, eptr=NULL, ws=NULL, wsb=0):
        return L.mla_sparse_fwd_ext(fake, 16 * 576, 576, fake, 656, 10, fake, fake, 8, extra, 656, 10, eptr, fake, 4,
                                    NULL, splits, 0.1, 1, fake, 16 * 512, 512, NULL, 4, 16, ws, wsb, NULL)
    assert ext(splits=0) == -2 and ext(splits=65) == -2
    assert ext(extra=fake) == -1                 # a second segment without its indptr
    assert ext() == -1                           # kv_splits = 2 needs a workspace
    assert b"workspace" in L.mla_last_error()

    assert L.mla_absorb_q(fake, 16 * 128, 128, fake, fake, 16 * 512, 512, 4, 16, 100, NULL) == -2   # P not 64k
    assert L.mla_absorb_q(fake, 16 * 128, 128, fake, fake, 16 * 512, 512, 0, 16, 128, NULL) == 0
    assert L.mla_v_up_proj(fake, 16 * 512, 512, fake, NULL, 0, fake, 16 * 100, 100, 4, 16, 100, NULL) == -2  # V
    assert L.mla_v_up_proj(fake, 16 * 512, 512, ctypes.c_void_p((1 << 20) + 2), NULL, 0, fake, 16 * 128, 128, 4, 16,
                           128, NULL) == -1      # weights not 16-byte aligned


def test_test_aids_are_exported(L):
    L.mla_debug_stall_next_decode(0)            # disarms: no GPU work
    assert hasattr(L, "mla_sparse_fwd_staged")
