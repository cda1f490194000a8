"""MLA over the 576-wide latent KV cache on GB300 (sm_103a): Python binding of libmla.

The functions here only marshal torch tensors (device memory, strides, the current CUDA
stream) into the C ABI of ``include/mla.h``; every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if ``libmla.so`` is missing or fails to load,
importing the binding raises.

Entry points (same names as the C ABI, without the ``mla_`` prefix):

  q_concat_cache_insert  decode epilogue: mqa_q = [ql_nope | q_pe] (+ GPT-J RoPE), latent
                         insert into a bf16 / plain fp8 / fp8_ds_mla paged cache
  sparse_fwd             sparse CSR forward over 656-byte fp8_ds_mla records
  paged_decode           paged decode / spec-verify (split-K + LSE merge)
  gather_dequant         paged entries -> exact fp32 values (test aid)
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

CACHE_BF16, CACHE_FP8, CACHE_FP8_DS_MLA = 0, 1, 2
ENTRY_BYTES = {CACHE_BF16: 1152, CACHE_FP8: 576, CACHE_FP8_DS_MLA: 656}
_FMT_NAMES = {"bf16": CACHE_BF16, "auto": CACHE_BF16, "fp8": CACHE_FP8, "fp8_ds_mla": CACHE_FP8_DS_MLA}

_lib = None


class MLAError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libmla.so (build it first with ``build.build()``).  Raises if it is missing."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise ImportError(f"libmla.so not built ({path}); run mla_latent_cache_attention_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        L.mla_last_error.restype = ctypes.c_char_p
        L.mla_version.restype = ctypes.c_char_p
        L.mla_read_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        L.mla_q_concat_cache_insert.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, vp, i64, vp, vp, i32,
                                                i64, i64, i64, i32, vp, vp, vp, vp, vp, i64, i32, i32, vp]
        L.mla_sparse_fwd.argtypes = [vp, i64, i64, vp, i64, i64, vp, vp, i64, f32, i32, vp, i64, i64, vp,
                                     i32, i32, vp]
        L.mla_paged_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.mla_paged_decode_workspace_size.restype = sz
        L.mla_paged_decode.argtypes = [vp, i64, i64, vp, i32, i64, i64, i64, i32, vp, i64, vp, i32, i32, i32,
                                       i32, f32, f32, f32, vp, i64, i64, vp, vp, sz, vp]
        L.mla_paged_decode_noalloc.argtypes = [vp, i64, i64, vp, i32, i64, i64, i64, i32, vp, i64, vp, i32, i32,
                                               i32, i32, f32, f32, f32, vp, i64, i64, vp, vp]
        L.mla_paged_decode_noalloc.restype = ctypes.c_int
        L.mla_profile_attention_events.argtypes = [vp, vp]
        L.mla_profile_attention_events.restype = None
        L.mla_gather_dequant.argtypes = [vp, i32, i64, i64, i64, i32, vp, i64, vp, vp]
        for f in ("mla_q_concat_cache_insert", "mla_sparse_fwd", "mla_paged_decode", "mla_gather_dequant"):
            getattr(L, f).restype = ctypes.c_int
        L.mla_read_device_errors.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int):
    if rc != 0:
        raise MLAError(f"libmla error {rc}: {lib().mla_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return _FMT_NAMES[fmt]
    return int(fmt)


def _cache_geometry(kv_cache: torch.Tensor):
    """[num_blocks, block_size, entry_stride] view of a paged cache (any 1- or 2-byte dtype)."""
    es = kv_cache.element_size()
    if kv_cache.dim() == 4:      # [nb, 1, bs, entry] (a head axis of size 1)
        kv_cache = kv_cache.squeeze(1)
    assert kv_cache.dim() == 3 and kv_cache.stride(2) == 1, "cache must be [num_blocks, block_size, entry]"
    return kv_cache.shape[0], kv_cache.stride(0) * es, kv_cache.stride(1) * es, kv_cache.shape[1]


def version() -> str:
    return lib().mla_version().decode()


def profile_attention_events(start=None, stop=None):
    """Bracket later attention-kernel launches of this thread with two torch.cuda.Events
    (recorded on the call's stream); ``None, None`` turns it off."""
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    lib().mla_profile_attention_events(h(start), h(stop))


def read_device_errors(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error word."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    v = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        _check(lib().mla_read_device_errors(ctypes.byref(v),
                                            ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)))
    return int(v.value)


def q_concat_cache_insert(ql_nope, q_pe, kv_c_normed, k_pe, kv_cache, slot_mapping, *, fmt,
                          q_scale_inv=None, cache_scale_inv=None, positions=None, cos_sin_cache=None,
                          mqa_q=None):
    """Decode epilogue.  Returns mqa_q [B, H, 576] (bf16, or uint8 E4M3 codes for fp8);
    writes kv_cache in place."""
    fmt = _fmt(fmt)
    k_pe = k_pe.reshape(k_pe.shape[0], -1)
    B, H, _ = ql_nope.shape
    if mqa_q is None:
        dt = torch.uint8 if fmt == CACHE_FP8 else torch.bfloat16
        mqa_q = torch.empty((B, H, 576), dtype=dt, device=ql_nope.device)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    max_pos = 0 if cos_sin_cache is None else cos_sin_cache.shape[0]
    _check(lib().mla_q_concat_cache_insert(
        _ptr(ql_nope), ql_nope.stride(0), ql_nope.stride(1), _ptr(q_pe), q_pe.stride(0), q_pe.stride(1),
        _ptr(kv_c_normed), kv_c_normed.stride(0), _ptr(k_pe), k_pe.stride(0), _ptr(mqa_q), _ptr(kv_cache),
        fmt, nb, bstride, estride, bs, _ptr(slot_mapping), _ptr(q_scale_inv), _ptr(cache_scale_inv),
        _ptr(positions), _ptr(cos_sin_cache), max_pos, B, H, _stream(ql_nope)))
    return mqa_q


def sparse_fwd(q, kv_records, kv_indptr, kv_indices, softmax_scale, *, has_invalid=False, out=None,
               return_lse=False, num_records=None):
    """Sparse forward over fp8_ds_mla records [N, >=656] (uint8).  Returns (out, lse)."""
    T, H, _ = q.shape
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=q.device) if return_lse else None
    rec = kv_records.reshape(-1, kv_records.shape[-1]) if kv_records.dim() != 2 else kv_records
    n_rec = rec.shape[0] if num_records is None else num_records
    _check(lib().mla_sparse_fwd(
        _ptr(q), q.stride(0), q.stride(1), _ptr(rec), rec.stride(0) * rec.element_size(), n_rec,
        _ptr(kv_indptr), _ptr(kv_indices), kv_indices.numel(), float(softmax_scale), int(bool(has_invalid)),
        _ptr(out), out.stride(0), out.stride(1), _ptr(lse), T, H, _stream(q)))
    return out, lse


def paged_decode_workspace_size(B, q_len, H, max_context, num_sms=0) -> int:
    return int(lib().mla_paged_decode_workspace_size(B, q_len, H, max_context, num_sms))


def paged_decode(q, kv_cache, block_table, seq_lens, *, fmt, q_len=1, max_context, softmax_scale,
                 q_scale=1.0, k_scale=1.0, out=None, return_lse=False, workspace=None):
    """Paged decode / spec-verify.  q [B*q_len, H, 576] (bf16, or uint8 E4M3 codes for fp8).
    Returns (out [B*q_len, H, 512] bf16, lse or None)."""
    fmt = _fmt(fmt)
    rows, H, _ = q.shape
    B = seq_lens.numel()
    assert rows == B * q_len, "q rows must be B * q_len"
    if out is None:
        out = torch.empty((rows, H, 512), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((rows, H), dtype=torch.float32, device=q.device) if return_lse else None
    need = paged_decode_workspace_size(B, q_len, H, max_context)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    _check(lib().mla_paged_decode(
        _ptr(q), q.stride(0), q.stride(1), _ptr(kv_cache), fmt, nb, bstride, estride, bs,
        _ptr(block_table), block_table.stride(0), _ptr(seq_lens), B, q_len, H, int(max_context),
        float(softmax_scale), float(q_scale), float(k_scale), _ptr(out), out.stride(0), out.stride(1),
        _ptr(lse), _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(q)))
    return out, lse


def gather_dequant(kv_cache, slots, *, fmt):
    """Exact fp32 values [n, 576] of the entries at `slots` (int64)."""
    fmt = _fmt(fmt)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    out = torch.empty((slots.numel(), 576), dtype=torch.float32, device=kv_cache.device)
    _check(lib().mla_gather_dequant(_ptr(kv_cache), fmt, nb, bstride, estride, bs, _ptr(slots),
                                    slots.numel(), _ptr(out), _stream(kv_cache)))
    return out
