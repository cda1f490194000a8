"""fp64 CPU oracle for MLA over the 576-wide latent cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding) never touches it,
and it shares no code with that path: the arithmetic lives in ``mla_oracle.c``, written
from the pages' definitions (see that file's header for the passages it follows and the
readings it takes where the pages are silent).

This module only compiles the C file (gcc, OpenMP, ``-ffp-contract=off``) and marshals
numpy arrays into it.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against values
the mathematics fixes (closed forms, invariants, library codecs, cross-API identities).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

BF16, FP8, DS_MLA = 0, 1, 2
ENTRY_BYTES = {BF16: 1152, FP8: 576, DS_MLA: 656}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmla_oracle.so`` (idempotent)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            vp, i64, i32, dbl, flt = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
            L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_double.restype = dbl
            L.orc_e4m3_from_float_sat.argtypes = [flt]
            L.orc_e4m3_from_float_sat.restype = ctypes.c_uint8
            L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_double.restype = dbl
            L.orc_bf16_from_float.argtypes = [flt]
            L.orc_bf16_from_float.restype = ctypes.c_uint16
            L.orc_decode_entry.argtypes = [i32, vp, vp]
            L.orc_sparse_fwd.argtypes = [vp, i64, i64, vp, i64, i64, vp, vp, dbl, i32, i32, i32, vp,
                                         i32, vp, vp]
            L.orc_sparse_fwd.restype = i32
            L.orc_paged_decode.argtypes = [i32, vp, i64, i64, vp, i64, i64, i64, i32, vp, i64, vp,
                                           i32, i32, i32, dbl, dbl, dbl, vp, i32, vp, vp]
            L.orc_paged_decode.restype = i32
            L.orc_merge.argtypes = [i32, vp, vp, vp, vp]
            L.orc_q_concat_cache_insert.argtypes = [i32, vp, i64, i64, vp, i64, i64, vp, i64, vp,
                                                    i64, vp, vp, i64, i64, i64, i32, vp, flt, flt,
                                                    vp, vp, i64, i32, i32]
            L.orc_q_concat_cache_insert.restype = i32
            L.orc_key_concat_cache_insert.argtypes = [i32, vp, i64, i64, vp, i64, i64, vp, i64, vp, i64, vp, vp,
                                                      i64, i64, i64, i32, vp, vp, vp, i64, i32, i32, i32]
            L.orc_key_concat_cache_insert.restype = i32
            L.orc_qkv_quant_cache_fp8_insert.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, vp, i64, vp, i64,
                                                         i64, vp, vp, vp, vp, i64, i64, i64, i32, vp, flt, flt,
                                                         flt, flt, vp, vp, i64, i32, i32, i32, i32]
            L.orc_qkv_quant_cache_fp8_insert.restype = i32
            L.orc_gather_context.argtypes = [i32, vp, i64, i64, i64, i32, vp, i64, vp, vp, i32, i64, i32, flt, vp,
                                             i64]
            L.orc_gather_context.restype = i32
            L.orc_merge_attn_states.argtypes = [vp, i64, i64, vp, vp, i64, i64, vp, i32, i32, i32, vp, vp]
            L.orc_merge_attn_states.restype = None
            L.orc_sparse_fwd_ext.argtypes = [vp, i64, i64, vp, i64, i64, vp, vp, vp, i64, i64, vp, vp, vp, dbl, i32,
                                             i32, i32, vp, vp]
            L.orc_sparse_fwd_ext.restype = i32
            L.orc_head_bmm.argtypes = [vp, i64, i64, vp, vp, i64, i32, i32, i32, i32, vp]
            L.orc_head_bmm.restype = None
            L.orc_ds_tile_exponent.argtypes = [dbl]
            L.orc_ds_tile_exponent.restype = i32
            L.orc_rope_fp32.argtypes = [vp, vp, vp]
            _lib = L
    return _lib


# ------------------------------------------------------------------------------------
# Codecs (scalar and vectorised through the C functions).
# ------------------------------------------------------------------------------------

def e4m3_to_f64(codes) -> np.ndarray:
    L = lib()
    table = np.array([L.orc_e4m3_to_double(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_from_f32(x) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    flat, of = x.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        of[i] = L.orc_e4m3_from_float_sat(float(flat[i]))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_from_f32(x) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat, of = x.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        of[i] = L.orc_bf16_from_float(float(flat[i]))
    return out


def decode_entry(fmt: int, entry_bytes) -> np.ndarray:
    e = np.ascontiguousarray(entry_bytes, dtype=np.uint8)
    assert e.size >= ENTRY_BYTES[fmt]
    out = np.empty(576, dtype=np.float64)
    lib().orc_decode_entry(fmt, _P(e), _P(out))
    return out


def ds_tile_exponent(amax: float) -> int:
    return int(lib().orc_ds_tile_exponent(float(amax)))


def rope_fp32(x, cs_row) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    cs = np.ascontiguousarray(cs_row, dtype=np.float32)
    y = np.empty(64, dtype=np.float32)
    lib().orc_rope_fp32(_P(x), _P(cs), _P(y))
    return y


# ------------------------------------------------------------------------------------
# The three computations.
# ------------------------------------------------------------------------------------

def sparse_fwd(q_bits, records, indptr, indices, softmax_scale, has_invalid, rows=None):
    """q_bits: uint16 [T, H, 576] (bf16 bits, last stride 1); records: uint8 [N, stride >= 656].

    Returns (out [n_rows, H, 512] f64, lse [n_rows, H] f64).  ``rows`` selects query rows.
    """
    q_bits = np.asarray(q_bits)
    assert q_bits.dtype == np.uint16 and q_bits.strides[2] == 2
    T, H, _ = q_bits.shape
    rec = np.asarray(records, dtype=np.uint8)
    assert rec.ndim == 2 and rec.strides[1] == 1 and rec.shape[1] >= 656
    indptr = np.ascontiguousarray(indptr, dtype=np.int64)
    indices = np.ascontiguousarray(indices, dtype=np.int64)
    if indices.size == 0:
        indices = np.zeros(1, dtype=np.int64)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = T if rows_a is None else rows_a.size
    out = np.zeros((n, H, 512), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    rc = lib().orc_sparse_fwd(_P(q_bits), q_bits.strides[0] // 2, q_bits.strides[1] // 2, _P(rec),
                              rec.strides[0], rec.shape[0], _P(indptr), _P(indices),
                              float(softmax_scale), int(bool(has_invalid)), T, H, _P(rows_a), n,
                              _P(out), _P(lse))
    if rc != 0:
        raise ValueError("oracle sparse_fwd: index out of range")
    return out, lse


def sparse_fwd_ext(q_bits, records, indptr, indices, softmax_scale, has_invalid, *, extra_records=None,
                   extra_indptr=None, extra_indices=None, attn_sink=None):
    """Sparse forward with the general op's extras: an attention sink per head (fp32 [H]) and a
    second key segment (extra_records [N2, >=656], extra_indptr [T+1], extra_indices).
    Returns (out [T, H, 512] f64, lse [T, H] f64)."""
    q_bits = np.asarray(q_bits)
    assert q_bits.dtype == np.uint16 and q_bits.strides[2] == 2
    T, H, _ = q_bits.shape
    rec = np.asarray(records, dtype=np.uint8)
    assert rec.ndim == 2 and rec.strides[1] == 1 and rec.shape[1] >= 656
    ip = np.ascontiguousarray(indptr, dtype=np.int64)
    ix = np.ascontiguousarray(indices, dtype=np.int64)
    if ix.size == 0:
        ix = np.zeros(1, dtype=np.int64)
    rec2 = ip2 = ix2 = None
    if extra_records is not None:
        rec2 = np.asarray(extra_records, dtype=np.uint8)
        assert rec2.ndim == 2 and rec2.strides[1] == 1 and rec2.shape[1] >= 656
        ip2 = np.ascontiguousarray(extra_indptr, dtype=np.int64)
        ix2 = np.ascontiguousarray(extra_indices, dtype=np.int64)
        if ix2.size == 0:
            ix2 = np.zeros(1, dtype=np.int64)
    sk = None if attn_sink is None else np.ascontiguousarray(attn_sink, dtype=np.float32)
    assert sk is None or sk.shape == (H,)
    out = np.zeros((T, H, 512), dtype=np.float64)
    lse = np.zeros((T, H), dtype=np.float64)
    rc = lib().orc_sparse_fwd_ext(_P(q_bits), q_bits.strides[0] // 2, q_bits.strides[1] // 2, _P(rec), rec.strides[0],
                                  rec.shape[0], _P(ip), _P(ix), _P(rec2), 0 if rec2 is None else rec2.strides[0],
                                  0 if rec2 is None else rec2.shape[0], _P(ip2), _P(ix2), _P(sk), float(softmax_scale),
                                  int(bool(has_invalid)), T, H, _P(out), _P(lse))
    if rc != 0:
        raise ValueError("oracle sparse_fwd_ext: index out of range")
    return out, lse


def paged_decode(fmt, q_bytes, cache, block_table, seq_lens, q_len, softmax_scale,
                 q_scale=1.0, k_scale=1.0, rows=None, *, block_stride=None, entry_stride=None):
    """q_bytes: uint8 [B*q_len, H, 576*elt] (bf16 bits as bytes, or e4m3 codes).

    cache: uint8 [num_blocks, block_size, entry_stride] (or pass explicit strides).
    Returns (out [n_rows, H, 512] f64, lse [n_rows, H] f64).
    """
    q_bytes = np.asarray(q_bytes)
    assert q_bytes.dtype == np.uint8 and q_bytes.ndim == 3
    rows_total, H, _ = q_bytes.shape
    cache = np.asarray(cache)
    assert cache.dtype == np.uint8 and cache.ndim == 3
    nb, bs, _ = cache.shape
    bstride = cache.strides[0] if block_stride is None else block_stride
    estride = cache.strides[1] if entry_stride is None else entry_stride
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = sl.size
    assert rows_total == B * q_len
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = rows_total if rows_a is None else rows_a.size
    out = np.zeros((n, H, 512), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    rc = lib().orc_paged_decode(int(fmt), _P(q_bytes), q_bytes.strides[0], q_bytes.strides[1],
                                _P(cache), nb, bstride, estride, bs, _P(bt), bt.shape[1], _P(sl),
                                B, q_len, H, float(softmax_scale), float(q_scale), float(k_scale),
                                _P(rows_a), n, _P(out), _P(lse))
    if rc != 0:
        raise ValueError("oracle paged_decode: block id out of range")
    return out, lse


def merge(parts, lse_parts):
    parts = np.ascontiguousarray(parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S = lse_parts.size
    assert parts.shape == (S, 512)
    out = np.zeros(512, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib().orc_merge(S, _P(parts), _P(lse_parts), _P(out), _P(lse))
    return out, float(lse[0])


def q_concat_cache_insert(fmt, ql_nope, q_pe, kv_c, k_pe, cache, slot_mapping, *,
                          q_scale_inv=1.0, cache_scale_inv=1.0, positions=None, cos_sin=None):
    """All activations are uint16 bf16 bits.  ``cache`` (uint8 [nb, bs, stride]) is updated
    in place; returns mqa_q (uint16 [B,H,576] bits, or uint8 e4m3 codes for plain fp8)."""
    ql_nope, q_pe = np.asarray(ql_nope), np.asarray(q_pe)
    kv_c, k_pe = np.asarray(kv_c), np.asarray(k_pe).reshape(np.asarray(k_pe).shape[0], -1)
    for a in (ql_nope, q_pe, kv_c, k_pe):
        assert a.dtype == np.uint16 and a.strides[-1] == 2
    B, H, _ = ql_nope.shape
    assert cache.dtype == np.uint8 and cache.ndim == 3 and cache.flags.writeable
    nb, bs, _ = cache.shape
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    if (positions is None) != (cos_sin is None):
        raise ValueError("positions and cos_sin must be given together")
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int64)
    cs = None if cos_sin is None else np.ascontiguousarray(cos_sin, dtype=np.float32)
    maxp = 0 if cs is None else cs.shape[0]
    if fmt == FP8:
        mqa = np.zeros((B, H, 576), dtype=np.uint8)
    else:
        mqa = np.zeros((B, H, 576), dtype=np.uint16)
    rc = lib().orc_q_concat_cache_insert(
        int(fmt), _P(ql_nope), ql_nope.strides[0] // 2, ql_nope.strides[1] // 2, _P(q_pe),
        q_pe.strides[0] // 2, q_pe.strides[1] // 2, _P(kv_c), kv_c.strides[0] // 2, _P(k_pe),
        k_pe.strides[0] // 2, _P(mqa), _P(cache), nb, cache.strides[0], cache.strides[1], bs,
        _P(sm), float(q_scale_inv), float(cache_scale_inv), _P(pos), _P(cs), maxp, B, H)
    if rc != 0:
        raise ValueError("oracle q_concat_cache_insert: slot or position out of range")
    return mqa


def _bits16(a, name):
    a = np.asarray(a)
    assert a.dtype == np.uint16 and a.strides[-1] == 2, f"{name}: uint16 bf16 bits with a unit last stride"
    return a


def _rope_args(positions, cos_sin):
    if (positions is None) != (cos_sin is None):
        raise ValueError("positions and cos_sin must be given together")
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int64)
    cs = None if cos_sin is None else np.ascontiguousarray(cos_sin, dtype=np.float32)
    return pos, cs, (0 if cs is None else cs.shape[0])


def key_concat_cache_insert(fmt, q, k_nope, k_pe, kv_c, cache, slot_mapping, *, positions=None, cos_sin=None):
    """Prefill epilogue for the bf16 (fmt=BF16) or fp8_ds_mla (fmt=DS_MLA) cache.  All
    activations are uint16 bf16 bits; ``q`` [Tp, H, dn+64] is rotated in place (when RoPE is
    on) and ``cache`` (uint8 [nb, bs, stride]) is updated in place.  Returns k_out (uint16
    [Tp, H, dn+64])."""
    assert fmt in (BF16, DS_MLA)
    q = _bits16(q, "q")
    assert q.flags.writeable
    k_nope = _bits16(k_nope, "k_nope")
    k_pe = _bits16(np.asarray(k_pe).reshape(np.asarray(k_pe).shape[0], -1), "k_pe")
    kv_c = _bits16(kv_c, "kv_c")
    Tp, H, dn = k_nope.shape
    assert q.shape == (Tp, H, dn + 64)
    assert cache.dtype == np.uint8 and cache.ndim == 3 and cache.flags.writeable
    nb, bs, _ = cache.shape
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    pos, cs, maxp = _rope_args(positions, cos_sin)
    k_out = np.zeros((Tp, H, dn + 64), dtype=np.uint16)
    rc = lib().orc_key_concat_cache_insert(
        int(fmt), _P(q), q.strides[0] // 2, q.strides[1] // 2, _P(k_nope), k_nope.strides[0] // 2,
        k_nope.strides[1] // 2, _P(k_pe), k_pe.strides[0] // 2, _P(kv_c), kv_c.strides[0] // 2, _P(k_out),
        _P(cache), nb, cache.strides[0], cache.strides[1], bs, _P(sm), _P(pos), _P(cs), maxp, Tp, H, dn)
    if rc != 0:
        raise ValueError("oracle key_concat_cache_insert: slot or position out of range")
    return k_out


def qkv_quant_cache_fp8_insert(q, k_nope, k_pe, kv_c, v, cache, slot_mapping, *, q_scale_inv, k_scale_inv,
                               v_scale_inv, cache_scale_inv, positions=None, cos_sin=None):
    """Prefill epilogue for the plain fp8 cache.  Returns (q_fp8, k_fp8, v_fp8) as uint8 E4M3
    codes; ``cache`` (uint8 [nb, bs, stride]) is updated in place; q is not modified."""
    q = _bits16(q, "q")
    k_nope = _bits16(k_nope, "k_nope")
    k_pe = _bits16(np.asarray(k_pe).reshape(np.asarray(k_pe).shape[0], -1), "k_pe")
    kv_c = _bits16(kv_c, "kv_c")
    v = _bits16(v, "v")
    Tp, H, dn = k_nope.shape
    dv = v.shape[2]
    assert q.shape == (Tp, H, dn + 64) and v.shape[:2] == (Tp, H)
    assert cache.dtype == np.uint8 and cache.ndim == 3 and cache.flags.writeable
    nb, bs, _ = cache.shape
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    pos, cs, maxp = _rope_args(positions, cos_sin)
    q8 = np.zeros((Tp, H, dn + 64), dtype=np.uint8)
    k8 = np.zeros((Tp, H, dn + 64), dtype=np.uint8)
    v8 = np.zeros((Tp, H, dv), dtype=np.uint8)
    rc = lib().orc_qkv_quant_cache_fp8_insert(
        _P(q), q.strides[0] // 2, q.strides[1] // 2, _P(k_nope), k_nope.strides[0] // 2, k_nope.strides[1] // 2,
        _P(k_pe), k_pe.strides[0] // 2, _P(kv_c), kv_c.strides[0] // 2, _P(v), v.strides[0] // 2,
        v.strides[1] // 2, _P(q8), _P(k8), _P(v8), _P(cache), nb, cache.strides[0], cache.strides[1], bs, _P(sm),
        float(q_scale_inv), float(k_scale_inv), float(v_scale_inv), float(cache_scale_inv), _P(pos), _P(cs), maxp,
        Tp, H, dn, dv)
    if rc != 0:
        raise ValueError("oracle qkv_quant_cache_fp8_insert: slot or position out of range")
    return q8, k8, v8


def gather_context(fmt, cache, block_table, cu_seq_lens, seq_starts=None, *, num_tokens=None, raw=False,
                   scale=1.0):
    """Chunk gather of paged context entries.  cache: uint8 [nb, bs, stride].  Returns uint16
    bf16 bits [num_tokens, 576] (raw=False) or uint8 entry bytes [num_tokens, entry] (raw=True);
    rows past cu_seq_lens[-1] stay zero."""
    cache = np.asarray(cache)
    assert cache.dtype == np.uint8 and cache.ndim == 3
    nb, bs, _ = cache.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seq_lens, dtype=np.int32)
    ss = None if seq_starts is None else np.ascontiguousarray(seq_starts, dtype=np.int32)
    batch = cu.size - 1
    n = int(cu[-1]) if num_tokens is None else int(num_tokens)
    if raw:
        dst = np.zeros((max(n, 1), ENTRY_BYTES[fmt]), dtype=np.uint8)
        row = dst.strides[0]
    else:
        dst = np.zeros((max(n, 1), 576), dtype=np.uint16)
        row = 576
    rc = lib().orc_gather_context(int(fmt), _P(cache), nb, cache.strides[0], cache.strides[1], bs, _P(bt),
                                  bt.shape[1], _P(cu), _P(ss), batch, n, 1 if raw else 0, float(scale), _P(dst), row)
    if rc != 0:
        raise ValueError("oracle gather_context: block id out of range")
    return dst[:n]


def merge_attn_states(prefix, prefix_lse, suffix, suffix_lse):
    """prefix / suffix: uint16 bf16 bits [T, H, D] (last stride 1); lse: fp32 [H, T].
    Returns (out fp64 [T, H, D], lse fp64 [H, T])."""
    prefix, suffix = np.asarray(prefix), np.asarray(suffix)
    assert prefix.dtype == np.uint16 and suffix.dtype == np.uint16
    assert prefix.strides[2] == 2 and suffix.strides[2] == 2
    T, H, D = prefix.shape
    assert suffix.shape == (T, H, D) and D <= 512
    pl = np.ascontiguousarray(prefix_lse, dtype=np.float32)
    sl = np.ascontiguousarray(suffix_lse, dtype=np.float32)
    assert pl.shape == (H, T) and sl.shape == (H, T)
    out = np.zeros((T, H, D), dtype=np.float64)
    lse = np.zeros((H, T), dtype=np.float64)
    lib().orc_merge_attn_states(_P(prefix), prefix.strides[0] // 2, prefix.strides[1] // 2, _P(pl), _P(suffix),
                                suffix.strides[0] // 2, suffix.strides[1] // 2, _P(sl), T, H, D, _P(out), _P(lse))
    return out, lse


def head_bmm(x, w, gate=None):
    """y[b, h, f] = sum_k x[b, h, k] w[h, k, f] (times sigmoid(gate[b, h*F + f]) when a gate is
    given), exact in fp64.  x: uint16 bf16 bits [B, H, K] (last stride 1); w: uint16 [H, K, F];
    gate: uint16 [B, H*F] (last stride 1) or None.  Returns fp64 [B, H, F]."""
    x = np.asarray(x)
    assert x.dtype == np.uint16 and x.strides[2] == 2
    w = np.ascontiguousarray(w, dtype=np.uint16)
    B, H, K = x.shape
    assert w.shape[:2] == (H, K)
    F = w.shape[2]
    g = None
    if gate is not None:
        g = np.asarray(gate)
        assert g.dtype == np.uint16 and g.strides[1] == 2 and g.shape == (B, H * F)
    y = np.zeros((B, H, F), dtype=np.float64)
    lib().orc_head_bmm(_P(x), x.strides[0] // 2, x.strides[1] // 2, _P(w), _P(g), 0 if g is None else g.strides[0] // 2,
                       B, H, K, F, _P(y))
    return y
