"""MLA over the 576-wide latent KV cache on GB300 (sm_103a): Python binding of libmla.

The functions here only marshal torch tensors (device memory, strides, the current CUDA
stream) into the C ABI of ``include/mla.h``; every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if ``libmla.so`` is missing or fails to load,
importing the binding raises.

Entry points (same names as the C ABI, without the ``mla_`` prefix):

  q_concat_cache_insert  decode epilogue: mqa_q = [ql_nope | q_pe] (+ GPT-J RoPE), latent
                         insert into a bf16 / plain fp8 / fp8_ds_mla paged cache
  key_concat_cache_insert   prefill epilogue (bf16 / fp8_ds_mla cache): full key
                         [k_nope | rope(k_pe)], q RoPE in place, latent insert
  qkv_quant_cache_fp8_insert  prefill epilogue (plain fp8 cache): E4M3 q / k / v with their
                         own scales, latent insert with the cache scale
  sparse_fwd             sparse CSR forward over 656-byte fp8_ds_mla records
  paged_decode           paged decode / spec-verify (split-K + LSE merge)
  absorb_q               BMM1: q_nope . W_UK_T per head -> ql_nope (latent query)
  v_up_proj              latent output . W_UV per head (+ sigmoid output gate)
  gather_context         chunked-context gather of paged entries (bf16 values or stored bytes)
  merge_attn_states      prefix / suffix merge of partial attentions by their LSEs
  gather_dequant         paged entries -> exact fp32 values (test aid)

Every tensor argument is checked here before the call (CUDA device, dtype, rank, unit
innermost stride; index tensors contiguous), so that a wrong tensor raises instead of being
read with the wrong layout.  Sparse indices may be int32 or int64.
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
        L.mla_sparse_fwd_staged.argtypes = L.mla_sparse_fwd.argtypes
        L.mla_sparse_fwd_ext_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.mla_sparse_fwd_ext_workspace_size.restype = sz
        L.mla_sparse_fwd_ext.argtypes = [vp, i64, i64, vp, i64, i64, vp, vp, i64, vp, i64, i64, vp, vp, i64, vp, i32,
                                         f32, i32, vp, i64, i64, vp, i32, i32, vp, sz, vp]
        L.mla_absorb_q.argtypes = [vp, i64, i64, vp, vp, i64, i64, i32, i32, i32, vp]
        L.mla_v_up_proj.argtypes = [vp, i64, i64, vp, vp, i64, vp, i64, i64, i32, i32, i32, vp]
        L.mla_gather_context.argtypes = [vp, i32, i64, i64, i64, i32, vp, i64, vp, vp, i32, i64, i32, f32, vp, i64, vp]
        L.mla_merge_attn_states.argtypes = [vp, i64, i64, vp, vp, i64, i64, vp, vp, i64, i64, vp, i32, i32, i32, vp]
        L.mla_key_concat_cache_insert.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, vp, i64, vp, vp, i32, i64, i64,
                                                  i64, i32, vp, vp, vp, i64, i32, i32, i32, vp]
        L.mla_qkv_quant_cache_fp8_insert.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, vp, i64, vp, i64, i64, vp,
                                                     vp, vp, vp, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, i64,
                                                     i32, i32, i32, i32, vp]
        L.mla_debug_stall_next_decode.argtypes = [i32]
        L.mla_debug_stall_next_decode.restype = None
        L.mla_debug_ds_cluster.argtypes = [i32]
        L.mla_debug_ds_cluster.restype = None
        for f in ("mla_q_concat_cache_insert", "mla_sparse_fwd", "mla_sparse_fwd_staged", "mla_paged_decode",
                  "mla_gather_dequant", "mla_key_concat_cache_insert", "mla_qkv_quant_cache_fp8_insert",
                  "mla_gather_context", "mla_merge_attn_states", "mla_sparse_fwd_ext", "mla_absorb_q",
                  "mla_v_up_proj"):
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


_BYTE_TYPES = (torch.uint8, torch.int8)
_INT32_MAX = 2 ** 31 - 1


def _need(t, name, dtypes, device, *, ndim=None, contiguous=False, inner=True):
    """Marshalling check of one tensor argument: a CUDA tensor on `device` of one of `dtypes`,
    with `ndim` dimensions, unit innermost stride (inner) or fully contiguous."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {', '.join(str(d) for d in dtypes)}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if inner and t.dim() > 0 and t.stride(-1) != 1 and t.shape[-1] > 1:
        raise ValueError(f"{name} must have a unit innermost stride")
    return t


def _cuda_device(t) -> torch.device:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    return t.device


def _index_i32(t, name, device, lo, hi):
    """int32 index tensor for the C ABI.  int64 input (accepted by the sparse forward's
    interface) is narrowed on the device after clamping to [lo, hi], so an id outside int32
    keeps its meaning: below lo stays masked / flagged, above hi stays out of range."""
    _need(t, name, (torch.int32, torch.int64), device, ndim=1, contiguous=True)
    if t.dtype == torch.int64:
        t = t.clamp(lo, hi).to(torch.int32)
    return t


def _cache_geometry(kv_cache: torch.Tensor):
    """[num_blocks, block_size, entry_stride] view of a paged cache (any 1- or 2-byte dtype)."""
    es = kv_cache.element_size()
    if kv_cache.dim() == 4 and kv_cache.shape[1] == 1:      # [nb, 1, bs, entry] (a head axis of size 1)
        kv_cache = kv_cache.squeeze(1)
    if kv_cache.dim() != 3 or kv_cache.stride(2) != 1:
        raise ValueError("kv_cache must be [num_blocks, block_size, entry] with a unit innermost stride")
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
    dev = _cuda_device(ql_nope)
    bf = (torch.bfloat16,)
    _need(ql_nope, "ql_nope", bf, dev, ndim=3)
    _need(q_pe, "q_pe", bf, dev, ndim=3)
    _need(kv_c_normed, "kv_c_normed", bf, dev, ndim=2)
    k_pe = _need(k_pe, "k_pe", bf, dev).reshape(k_pe.shape[0], -1)
    _need(slot_mapping, "slot_mapping", (torch.int64,), dev, ndim=1, contiguous=True)
    if positions is not None:
        _need(positions, "positions", (torch.int64,), dev, ndim=1, contiguous=True)
    if cos_sin_cache is not None:
        _need(cos_sin_cache, "cos_sin_cache", (torch.float32,), dev, ndim=2, contiguous=True)
    for n, t in (("q_scale_inv", q_scale_inv), ("cache_scale_inv", cache_scale_inv)):
        if t is not None:
            _need(t, n, (torch.float32,), dev)
    B, H, _ = ql_nope.shape
    if mqa_q is None:
        dt = torch.uint8 if fmt == CACHE_FP8 else torch.bfloat16
        mqa_q = torch.empty((B, H, 576), dtype=dt, device=dev)
    _need(mqa_q, "mqa_q", _BYTE_TYPES if fmt == CACHE_FP8 else bf, dev, ndim=3, contiguous=True)
    _need(kv_cache, "kv_cache", _BYTE_TYPES + bf, dev)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    max_pos = 0 if cos_sin_cache is None else cos_sin_cache.shape[0]
    with torch.cuda.device(dev):
        _check(lib().mla_q_concat_cache_insert(
            _ptr(ql_nope), ql_nope.stride(0), ql_nope.stride(1), _ptr(q_pe), q_pe.stride(0), q_pe.stride(1),
            _ptr(kv_c_normed), kv_c_normed.stride(0), _ptr(k_pe), k_pe.stride(0), _ptr(mqa_q), _ptr(kv_cache),
            fmt, nb, bstride, estride, bs, _ptr(slot_mapping), _ptr(q_scale_inv), _ptr(cache_scale_inv),
            _ptr(positions), _ptr(cos_sin_cache), max_pos, B, H, _stream(ql_nope)))
    return mqa_q


def _prefill_common(q, k_nope, k_pe, kv_c_normed, slot_mapping, positions, cos_sin_cache):
    dev = _cuda_device(q)
    bf = (torch.bfloat16,)
    _need(q, "q", bf, dev, ndim=3)
    _need(k_nope, "k_nope", bf, dev, ndim=3)
    k_pe = _need(k_pe, "k_pe", bf, dev).reshape(k_pe.shape[0], -1)
    _need(kv_c_normed, "kv_c_normed", bf, dev, ndim=2)
    _need(slot_mapping, "slot_mapping", (torch.int64,), dev, ndim=1, contiguous=True)
    if positions is not None:
        _need(positions, "positions", (torch.int64,), dev, ndim=1, contiguous=True)
    if cos_sin_cache is not None:
        _need(cos_sin_cache, "cos_sin_cache", (torch.float32,), dev, ndim=2, contiguous=True)
    Tp, H, dn = k_nope.shape
    if q.shape != (Tp, H, dn + 64):
        raise ValueError(f"q must be [Tp, H, dn + 64] = {(Tp, H, dn + 64)}, got {tuple(q.shape)}")
    return dev, k_pe, Tp, H, dn


def key_concat_cache_insert(q, k_nope, k_pe, kv_c_normed, kv_cache, slot_mapping, *, fmt, positions=None,
                            cos_sin_cache=None, k_out=None):
    """Prefill epilogue for the bf16 / fp8_ds_mla cache.  Rotates the rope part of q in place
    (when positions are given), writes kv_cache in place and returns k_out [Tp, H, dn + 64]."""
    fmt = _fmt(fmt)
    dev, k_pe, Tp, H, dn = _prefill_common(q, k_nope, k_pe, kv_c_normed, slot_mapping, positions, cos_sin_cache)
    if k_out is None:
        k_out = torch.empty((Tp, H, dn + 64), dtype=torch.bfloat16, device=dev)
    _need(k_out, "k_out", (torch.bfloat16,), dev, ndim=3, contiguous=True)
    _need(kv_cache, "kv_cache", _BYTE_TYPES + (torch.bfloat16,), dev)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    max_pos = 0 if cos_sin_cache is None else cos_sin_cache.shape[0]
    with torch.cuda.device(dev):
        _check(lib().mla_key_concat_cache_insert(
            _ptr(q), q.stride(0), q.stride(1), _ptr(k_nope), k_nope.stride(0), k_nope.stride(1), _ptr(k_pe),
            k_pe.stride(0), _ptr(kv_c_normed), kv_c_normed.stride(0), _ptr(k_out), _ptr(kv_cache), fmt, nb, bstride,
            estride, bs, _ptr(slot_mapping), _ptr(positions), _ptr(cos_sin_cache), max_pos, Tp, H, dn, _stream(q)))
    return k_out


def qkv_quant_cache_fp8_insert(q, k_nope, k_pe, kv_c_normed, v, kv_cache, slot_mapping, *, q_scale_inv, k_scale_inv,
                               v_scale_inv, cache_scale_inv, positions=None, cos_sin_cache=None):
    """Prefill epilogue for the plain fp8 cache.  Returns (q_fp8, k_fp8, v_fp8) as uint8 E4M3
    codes; writes kv_cache in place.  The four scales are device fp32 scalars (1 / scale)."""
    dev, k_pe, Tp, H, dn = _prefill_common(q, k_nope, k_pe, kv_c_normed, slot_mapping, positions, cos_sin_cache)
    _need(v, "v", (torch.bfloat16,), dev, ndim=3)
    dv = v.shape[2]
    for n, t in (("q_scale_inv", q_scale_inv), ("k_scale_inv", k_scale_inv), ("v_scale_inv", v_scale_inv),
                 ("cache_scale_inv", cache_scale_inv)):
        _need(t, n, (torch.float32,), dev)
    _need(kv_cache, "kv_cache", _BYTE_TYPES, dev)
    q8 = torch.empty((Tp, H, dn + 64), dtype=torch.uint8, device=dev)
    k8 = torch.empty((Tp, H, dn + 64), dtype=torch.uint8, device=dev)
    v8 = torch.empty((Tp, H, dv), dtype=torch.uint8, device=dev)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    max_pos = 0 if cos_sin_cache is None else cos_sin_cache.shape[0]
    with torch.cuda.device(dev):
        _check(lib().mla_qkv_quant_cache_fp8_insert(
            _ptr(q), q.stride(0), q.stride(1), _ptr(k_nope), k_nope.stride(0), k_nope.stride(1), _ptr(k_pe),
            k_pe.stride(0), _ptr(kv_c_normed), kv_c_normed.stride(0), _ptr(v), v.stride(0), v.stride(1), _ptr(q8),
            _ptr(k8), _ptr(v8), _ptr(kv_cache), nb, bstride, estride, bs, _ptr(slot_mapping), _ptr(q_scale_inv),
            _ptr(k_scale_inv), _ptr(v_scale_inv), _ptr(cache_scale_inv), _ptr(positions), _ptr(cos_sin_cache), max_pos,
            Tp, H, dn, dv, _stream(q)))
    return q8, k8, v8


def sparse_fwd(q, kv_records, kv_indptr, kv_indices, softmax_scale, *, has_invalid=False, out=None,
               return_lse=False, num_records=None, kernel="gather", attn_sink=None, extra_kv=None, extra_indptr=None,
               extra_indices=None, kv_splits=1, workspace=None, lse=None):
    """Sparse forward over fp8_ds_mla records [N, >=656] (uint8).  Returns (out, lse).

    kv_indptr / kv_indices may be int32 or int64 (int64 is narrowed on the device, keeping
    masked and out-of-range ids as such).  attn_sink (fp32 [H]), a second key segment
    (extra_kv records with extra_indptr / extra_indices) and kv_splits > 1 run
    mla_sparse_fwd_ext.  kernel="staged" runs the test aid mla_sparse_fwd_staged (the second
    kernel design) instead of mla_sparse_fwd."""
    dev = _cuda_device(q)
    _need(q, "q", (torch.bfloat16,), dev, ndim=3)
    _need(kv_records, "kv_records", _BYTE_TYPES, dev)
    T, H, _ = q.shape
    rec = kv_records.reshape(-1, kv_records.shape[-1]) if kv_records.dim() != 2 else kv_records
    n_rec = rec.shape[0] if num_records is None else num_records
    if kv_indptr.numel() != T + 1:
        raise ValueError(f"kv_indptr must have T + 1 = {T + 1} entries, got {kv_indptr.numel()}")
    n_idx = kv_indices.numel()
    kv_indptr = _index_i32(kv_indptr, "kv_indptr", dev, 0, min(n_idx, _INT32_MAX))
    kv_indices = _index_i32(kv_indices, "kv_indices", dev, -1, min(n_rec, _INT32_MAX))
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev, ndim=3)
    if return_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", (torch.float32,), dev, ndim=2, contiguous=True)
        if tuple(lse.shape) != (T, H):
            raise ValueError(f"lse must be [T, H] = {(T, H)}")
    ext = attn_sink is not None or extra_kv is not None or int(kv_splits) != 1
    if not ext:
        fn = {"gather": lib().mla_sparse_fwd, "staged": lib().mla_sparse_fwd_staged}[kernel]
        with torch.cuda.device(dev):
            _check(fn(
                _ptr(q), q.stride(0), q.stride(1), _ptr(rec), rec.stride(0) * rec.element_size(), n_rec,
                _ptr(kv_indptr), _ptr(kv_indices), n_idx, float(softmax_scale), int(bool(has_invalid)),
                _ptr(out), out.stride(0), out.stride(1), _ptr(lse), T, H, _stream(q)))
        return out, lse
    if kernel != "gather":
        raise ValueError("the sink, second segment and kv_splits are served by the gather kernel only")
    rec2, n_rec2, n_idx2 = None, 0, 0
    if extra_kv is not None:
        _need(extra_kv, "extra_kv", _BYTE_TYPES, dev)
        rec2 = extra_kv.reshape(-1, extra_kv.shape[-1]) if extra_kv.dim() != 2 else extra_kv
        n_rec2 = rec2.shape[0]
        if extra_indptr is None or extra_indices is None or extra_indptr.numel() != T + 1:
            raise ValueError("extra_kv needs extra_indptr [T + 1] and extra_indices")
        n_idx2 = extra_indices.numel()
        extra_indptr = _index_i32(extra_indptr, "extra_indptr", dev, 0, min(n_idx2, _INT32_MAX))
        extra_indices = _index_i32(extra_indices, "extra_indices", dev, -1, min(n_rec2, _INT32_MAX))
    if attn_sink is not None:
        _need(attn_sink, "attn_sink", (torch.float32,), dev, ndim=1, contiguous=True)
        if attn_sink.numel() != H:
            raise ValueError(f"attn_sink must have H = {H} entries")
    with torch.cuda.device(dev):
        need = int(lib().mla_sparse_fwd_ext_workspace_size(T, H, int(kv_splits), int(rec2 is not None),
                                                          int(attn_sink is not None)))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _check(lib().mla_sparse_fwd_ext(
            _ptr(q), q.stride(0), q.stride(1), _ptr(rec), rec.stride(0) * rec.element_size(), n_rec,
            _ptr(kv_indptr), _ptr(kv_indices), n_idx, _ptr(rec2), 0 if rec2 is None else rec2.stride(0), n_rec2,
            _ptr(extra_indptr) if rec2 is not None else None, _ptr(extra_indices) if rec2 is not None else None,
            n_idx2, _ptr(attn_sink), int(kv_splits), float(softmax_scale), int(bool(has_invalid)), _ptr(out),
            out.stride(0), out.stride(1), _ptr(lse), T, H, _ptr(workspace),
            0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(q)))
    return out, lse


def paged_decode_workspace_size(B, q_len, H, max_context, num_sms=0) -> int:
    return int(lib().mla_paged_decode_workspace_size(B, q_len, H, max_context, num_sms))


def paged_decode(q, kv_cache, block_table, seq_lens, *, fmt, q_len=1, max_context, softmax_scale,
                 q_scale=1.0, k_scale=1.0, out=None, return_lse=False, workspace=None, lse=None):
    """Paged decode / spec-verify.  q [B*q_len, H, 576] (bf16, or uint8 E4M3 codes for fp8).
    Returns (out [B*q_len, H, 512] bf16, lse or None)."""
    fmt = _fmt(fmt)
    dev = _cuda_device(q)
    _need(q, "q", _BYTE_TYPES if fmt == CACHE_FP8 else (torch.bfloat16,), dev, ndim=3)
    _need(kv_cache, "kv_cache", _BYTE_TYPES + (torch.bfloat16,), dev)
    _need(block_table, "block_table", (torch.int32,), dev, ndim=2)
    _need(seq_lens, "seq_lens", (torch.int32,), dev, ndim=1, contiguous=True)
    rows, H, _ = q.shape
    B = seq_lens.numel()
    if rows != B * q_len:
        raise ValueError(f"q has {rows} rows; expected B * q_len = {B * q_len}")
    if out is None:
        out = torch.empty((rows, H, 512), dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev, ndim=3)
    if return_lse and lse is None:
        lse = torch.empty((rows, H), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", (torch.float32,), dev, ndim=2, contiguous=True)
        if tuple(lse.shape) != (rows, H):
            raise ValueError(f"lse must be [B * q_len, H] = {(rows, H)}")
    with torch.cuda.device(dev):
        need = paged_decode_workspace_size(B, q_len, H, max_context)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if workspace is not None:
            _need(workspace, "workspace", _BYTE_TYPES, dev, contiguous=True)
        nb, bstride, estride, bs = _cache_geometry(kv_cache)
        _check(lib().mla_paged_decode(
            _ptr(q), q.stride(0), q.stride(1), _ptr(kv_cache), fmt, nb, bstride, estride, bs,
            _ptr(block_table), block_table.stride(0), _ptr(seq_lens), B, q_len, H, int(max_context),
            float(softmax_scale), float(q_scale), float(k_scale), _ptr(out), out.stride(0), out.stride(1),
            _ptr(lse), _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
            _stream(q)))
    return out, lse


def absorb_q(q_nope, w_uk_t, *, ql_nope=None):
    """BMM1: ql_nope[b, h] = q_nope[b, h] . w_uk_t[h]; q_nope bf16 [B, H, P] (unit innermost
    stride), w_uk_t bf16 [H, P, 512].  Returns ql_nope [B, H, 512] bf16."""
    dev = _cuda_device(q_nope)
    _need(q_nope, "q_nope", (torch.bfloat16,), dev, ndim=3)
    _need(w_uk_t, "w_uk_t", (torch.bfloat16,), dev, ndim=3, contiguous=True)
    B, H, P = q_nope.shape
    if tuple(w_uk_t.shape) != (H, P, 512):
        raise ValueError(f"w_uk_t must be [H, P, 512] = {(H, P, 512)}, got {tuple(w_uk_t.shape)}")
    if ql_nope is None:
        ql_nope = torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev)
    _need(ql_nope, "ql_nope", (torch.bfloat16,), dev, ndim=3)
    with torch.cuda.device(dev):
        _check(lib().mla_absorb_q(_ptr(q_nope), q_nope.stride(0), q_nope.stride(1), _ptr(w_uk_t), _ptr(ql_nope),
                                  ql_nope.stride(0), ql_nope.stride(1), B, H, P, _stream(q_nope)))
    return ql_nope


def v_up_proj(latent, w_uv, gate=None, *, out=None):
    """out[b, h] = latent[b, h] . w_uv[h] (times bf16(sigmoid(gate[b, h*V:(h+1)*V])) when a
    gate is given); latent bf16 [B, H, 512], w_uv bf16 [H, 512, V], gate bf16 [B, H * V].
    Returns out [B, H, V] bf16."""
    dev = _cuda_device(latent)
    _need(latent, "latent", (torch.bfloat16,), dev, ndim=3)
    _need(w_uv, "w_uv", (torch.bfloat16,), dev, ndim=3, contiguous=True)
    B, H, L = latent.shape
    if L != 512 or w_uv.shape[0] != H or w_uv.shape[1] != 512:
        raise ValueError("latent must be [B, H, 512] and w_uv [H, 512, V]")
    V = w_uv.shape[2]
    if gate is not None:
        _need(gate, "gate", (torch.bfloat16,), dev, ndim=2)
        if tuple(gate.shape) != (B, H * V):
            raise ValueError(f"gate must be [B, H * V] = {(B, H * V)}")
    if out is None:
        out = torch.empty((B, H, V), dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev, ndim=3)
    with torch.cuda.device(dev):
        _check(lib().mla_v_up_proj(_ptr(latent), latent.stride(0), latent.stride(1), _ptr(w_uv), _ptr(gate),
                                   0 if gate is None else gate.stride(0), _ptr(out), out.stride(0), out.stride(1), B, H,
                                   V, _stream(latent)))
    return out


def gather_context(kv_cache, block_table, cu_seq_lens, seq_starts=None, *, fmt, num_tokens, raw=False,
                   scale=1.0, dst=None):
    """Chunked-context gather: rows cu_seq_lens[b] .. cu_seq_lens[b+1]-1 hold request b's context
    positions seq_starts[b] + i.  Returns dst [num_tokens, 576] bf16 (raw=False) or
    [num_tokens, entry bytes] uint8 (raw=True)."""
    fmt = _fmt(fmt)
    dev = _cuda_device(kv_cache)
    _need(kv_cache, "kv_cache", _BYTE_TYPES + (torch.bfloat16,), dev)
    _need(block_table, "block_table", (torch.int32,), dev, ndim=2)
    _need(cu_seq_lens, "cu_seq_lens", (torch.int32,), dev, ndim=1, contiguous=True)
    if seq_starts is not None:
        _need(seq_starts, "seq_starts", (torch.int32,), dev, ndim=1, contiguous=True)
    batch = cu_seq_lens.numel() - 1
    if block_table.shape[0] < batch or (seq_starts is not None and seq_starts.numel() < batch):
        raise ValueError("block_table and seq_starts need a row per request of the chunk")
    if dst is None:
        dst = (torch.empty((num_tokens, ENTRY_BYTES[fmt]), dtype=torch.uint8, device=dev) if raw else
               torch.empty((num_tokens, 576), dtype=torch.bfloat16, device=dev))
    _need(dst, "dst", _BYTE_TYPES if raw else (torch.bfloat16,), dev, ndim=2)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    with torch.cuda.device(dev):
        _check(lib().mla_gather_context(_ptr(kv_cache), fmt, nb, bstride, estride, bs, _ptr(block_table),
                                        block_table.stride(0), _ptr(cu_seq_lens), _ptr(seq_starts), batch,
                                        int(num_tokens), 1 if raw else 0, float(scale), _ptr(dst),
                                        dst.stride(0) * dst.element_size(), _stream(kv_cache)))
    return dst


def merge_attn_states(prefix_output, prefix_lse, suffix_output, suffix_lse, *, output=None, return_lse=False):
    """Merge of a prefix and a suffix partial attention (bf16 [T, H, D], lse fp32 [H, T]).
    Returns (output [T, H, D] bf16, lse [H, T] or None)."""
    dev = _cuda_device(prefix_output)
    _need(prefix_output, "prefix_output", (torch.bfloat16,), dev, ndim=3)
    _need(suffix_output, "suffix_output", (torch.bfloat16,), dev, ndim=3)
    T, H, D = prefix_output.shape
    if tuple(suffix_output.shape) != (T, H, D):
        raise ValueError("prefix and suffix outputs differ in shape")
    for n, t in (("prefix_lse", prefix_lse), ("suffix_lse", suffix_lse)):
        _need(t, n, (torch.float32,), dev, ndim=2, contiguous=True)
        if tuple(t.shape) != (H, T):
            raise ValueError(f"{n} must be [H, T] = {(H, T)}, got {tuple(t.shape)}")
    if output is None:
        output = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    _need(output, "output", (torch.bfloat16,), dev, ndim=3)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev) if return_lse else None
    with torch.cuda.device(dev):
        _check(lib().mla_merge_attn_states(
            _ptr(output), output.stride(0), output.stride(1), _ptr(lse), _ptr(prefix_output), prefix_output.stride(0),
            prefix_output.stride(1), _ptr(prefix_lse), _ptr(suffix_output), suffix_output.stride(0),
            suffix_output.stride(1), _ptr(suffix_lse), T, H, D, _stream(prefix_output)))
    return output, lse


def gather_dequant(kv_cache, slots, *, fmt):
    """Exact fp32 values [n, 576] of the entries at `slots` (int64)."""
    fmt = _fmt(fmt)
    dev = _cuda_device(kv_cache)
    _need(slots, "slots", (torch.int64,), dev, ndim=1, contiguous=True)
    nb, bstride, estride, bs = _cache_geometry(kv_cache)
    out = torch.empty((slots.numel(), 576), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _check(lib().mla_gather_dequant(_ptr(kv_cache), fmt, nb, bstride, estride, bs, _ptr(slots),
                                        slots.numel(), _ptr(out), _stream(kv_cache)))
    return out


def debug_stall_next_decode(wait_us: int):
    """Test aid (mla_debug_stall_next_decode): the next page-kernel decode on this thread
    issues no loads and its waits give up after wait_us microseconds."""
    lib().mla_debug_stall_next_decode(int(wait_us))


def debug_ds_cluster(size: int = 0) -> None:
    """Test aid (mla_debug_ds_cluster): fp8_ds_mla decodes on this host thread run the head
    groups of a request as clusters of `size` CTAs (2, 3 or 6) that share each page tile, one
    CTA per group (1), or as the library chooses (0: pairs where the group count is even)."""
    lib().mla_debug_ds_cluster(int(size))
