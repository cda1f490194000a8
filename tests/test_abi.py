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
