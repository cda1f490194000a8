"""Seeded synthetic workloads for the MLA latent-cache path.

This module only draws random inputs (numpy ``default_rng``) and lays them out in the
byte formats the path reads; it contains none of the attention arithmetic.  Number-format
conversions of the random draws go through library casts (``torch`` CPU casts to bfloat16
and float8_e4m3fn) so that neither the oracle nor the CUDA library lends code to the other.

Large arrays are drawn through a 65536-level quantile table: a uniform 16-bit draw picks a
quantile of N(0, 1), which is then cast once.  This is N(0, 1) discretised at 2^-16 in the
CDF, and makes multi-GB caches cheap to generate on the host.

Workloads (all from the five benchmark configurations of the latent-cache path):
  0 tiny sparse forward          T=4, H=16, N=256 records, 64 indices per row
  1 paged bf16 decode + epilogue B=32, q=1, H=16, L ~ U[1024, 8192]
  2 sparse prefill               T=4096, H=16, N=65536, top-2048 per row
  3 fp8 spec-verify decode       B=64, q=4, H=16, L ~ U[16384, 131072]
  4 ds_mla large-batch decode    B=128, q=1, H=96, L ~ U[8192, 32768]
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16, FP8, DS_MLA = 0, 1, 2
ENTRY_BYTES = {BF16: 1152, FP8: 576, DS_MLA: 656}
SOFTMAX_SCALE = 192 ** -0.5

_QTABLES: dict = {}


def _normal_quantiles() -> np.ndarray:
    if "q" not in _QTABLES:
        from scipy.special import ndtri
        u = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
        _QTABLES["q"] = ndtri(u).astype(np.float32)
    return _QTABLES["q"]


def _bf16_bits_of(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _e4m3_codes_of(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(np.clip(x, -448.0, 448.0), dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def normal_bf16_bits(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) draws as bf16 bit patterns (uint16)."""
    key = "bf16"
    if key not in _QTABLES:
        _QTABLES[key] = _bf16_bits_of(_normal_quantiles())
    u = rng.integers(0, 65536, size=shape, dtype=np.uint16)
    return _QTABLES[key][u]


def normal_e4m3_codes(rng: np.random.Generator, shape, inv_scale: float) -> np.ndarray:
    """e4m3_sat(x * inv_scale) codes for x ~ N(0,1)."""
    key = ("e4m3", float(inv_scale))
    if key not in _QTABLES:
        _QTABLES[key] = _e4m3_codes_of(_normal_quantiles().astype(np.float64) * inv_scale)
    u = rng.integers(0, 65536, size=shape, dtype=np.uint16)
    return _QTABLES[key][u]


def finite_e4m3_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    """Bytes uniform over the 254 finite E4M3 codes (0x7F and 0xFF are NaN)."""
    r = rng.integers(0, 254, size=shape, dtype=np.uint8)
    return r + (r >= 0x7F).astype(np.uint8)


def ds_mla_records(rng: np.random.Generator, n: int, scale_lo=0.01, scale_hi=0.1) -> np.ndarray:
    """[n, 656] uint8 fp8_ds_mla records: 512 finite e4m3 | 4 fp32 scales U[lo,hi] | 64 bf16 N(0,1)."""
    rec = np.empty((n, 656), dtype=np.uint8)
    rec[:, :512] = finite_e4m3_bytes(rng, (n, 512))
    rec[:, 512:528] = rng.uniform(scale_lo, scale_hi, size=(n, 4)).astype(np.float32).view(np.uint8)
    rec[:, 528:656] = normal_bf16_bits(rng, (n, 64)).view(np.uint8)
    return rec


def cos_sin_table(max_position: int = 131072, rope: int = 64, base: float = 10000.0) -> np.ndarray:
    """[max_position, rope] fp32: columns 0..rope/2-1 cos(p*theta_i), the rest sin(p*theta_i),
    theta_i = base^(-2i/rope), evaluated in fp64 and rounded once to fp32."""
    key = ("cs", max_position, rope, base)
    if key not in _QTABLES:
        half = rope // 2
        theta = base ** (-2.0 * np.arange(half, dtype=np.float64) / rope)
        ang = np.arange(max_position, dtype=np.float64)[:, None] * theta[None, :]
        _QTABLES[key] = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    return _QTABLES[key]


# ------------------------------------------------------------------------------------
# Sparse forward workloads.
# ------------------------------------------------------------------------------------

@dataclass
class SparseCase:
    q: np.ndarray            # uint16 [T, H, 576] bf16 bits
    records: np.ndarray      # uint8 [N, 656]
    indptr: np.ndarray       # int32 [T+1]
    indices: np.ndarray      # int32 [nnz]
    softmax_scale: float
    has_invalid: bool
    return_lse: bool = True
    meta: dict = field(default_factory=dict)


def sparse_case(seed: int, T: int, H: int, N: int, per_row: int, p_invalid: float,
                replace: bool, empty_rows=(), ragged: bool = False,
                scale_lo=0.01, scale_hi=0.1) -> SparseCase:
    rng = np.random.default_rng(seed)
    q = normal_bf16_bits(rng, (T, H, 576))
    records = ds_mla_records(rng, N, scale_lo, scale_hi)
    lens = np.full(T, per_row, dtype=np.int64)
    if ragged:
        lens = rng.integers(0, per_row + 1, size=T)
    for r in empty_rows:
        lens[r] = 0
    indptr = np.zeros(T + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lens)
    idx = np.empty(int(indptr[-1]), dtype=np.int64)
    for t in range(T):
        n = int(lens[t])
        if n == 0:
            continue
        if replace:
            idx[indptr[t]:indptr[t + 1]] = rng.integers(0, N, size=n)
        else:
            idx[indptr[t]:indptr[t + 1]] = rng.choice(N, size=n, replace=False)
    if p_invalid > 0:
        idx[rng.random(idx.size) < p_invalid] = -1
    return SparseCase(q=q, records=records, indptr=indptr.astype(np.int32),
                      indices=idx.astype(np.int32), softmax_scale=SOFTMAX_SCALE,
                      has_invalid=p_invalid > 0, meta=dict(T=T, H=H, N=N, per_row=per_row))


def config0() -> SparseCase:
    """Tiny sparse forward: T=4, H=16, N=256, 64 indices per row (with replacement), ~10 %
    set to -1, row 3 empty; softmax_scale = 192^-0.5, lse returned; seed 0."""
    return sparse_case(0, T=4, H=16, N=256, per_row=64, p_invalid=0.10, replace=True,
                       empty_rows=(3,))


def config2(T: int = 4096, N: int = 65536, per_row: int = 2048) -> SparseCase:
    """Sparse prefill: T=4096, H=16, N=65536 records, 2048 indices per row uniform without
    replacement, ~5 % set to -1; seed 2."""
    return sparse_case(2, T=T, H=16, N=N, per_row=per_row, p_invalid=0.05, replace=False)


# ------------------------------------------------------------------------------------
# Paged decode workloads.
# ------------------------------------------------------------------------------------

@dataclass
class PagedCase:
    fmt: int
    q: np.ndarray            # uint8 [B*q_len, H, 576*elt] (bf16 bits as bytes, or e4m3 codes)
    cache: np.ndarray        # uint8 [num_blocks, block_size, entry_stride]
    block_table: np.ndarray  # int32 [B, max_blocks]
    seq_lens: np.ndarray     # int32 [B]
    q_len: int
    H: int
    max_context: int
    softmax_scale: float
    q_scale: float = 1.0
    k_scale: float = 1.0
    return_lse: bool = True
    meta: dict = field(default_factory=dict)


def _paged_layout(rng, B, L_lo, L_hi, block_size, max_context, seq_lens=None):
    if seq_lens is None:
        seq_lens = rng.integers(L_lo, L_hi + 1, size=B).astype(np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    nblk = (seq_lens + block_size - 1) // block_size
    total = int(nblk.sum())
    perm = rng.permutation(total).astype(np.int32)
    max_blocks = max(1, (max_context + block_size - 1) // block_size)
    bt = np.zeros((B, max_blocks), dtype=np.int32)
    o = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[o:o + nblk[b]]
        o += nblk[b]
    return seq_lens.astype(np.int32), bt, max(total, 1)


def paged_case(seed: int, fmt: int, B: int, q_len: int, H: int, L_lo: int, L_hi: int,
               block_size: int = 64, max_context: int | None = None, entry_pad: int = 0,
               q_scale: float = 1.0, k_scale: float = 1.0, seq_lens=None,
               return_lse: bool = True) -> PagedCase:
    rng = np.random.default_rng(seed)
    if max_context is None:
        max_context = int(L_hi if seq_lens is None else max(int(max(seq_lens)), 1))
    seq_lens, bt, nb = _paged_layout(rng, B, L_lo, L_hi, block_size, max_context, seq_lens)
    eb = ENTRY_BYTES[fmt]
    stride = eb + entry_pad
    cache = np.zeros((nb, block_size, stride), dtype=np.uint8)
    flat = cache.reshape(nb * block_size, stride)
    if fmt == BF16:
        flat[:, :eb] = normal_bf16_bits(rng, (nb * block_size, 576)).view(np.uint8)
    elif fmt == FP8:
        flat[:, :eb] = normal_e4m3_codes(rng, (nb * block_size, 576), 1.0 / k_scale)
    else:
        flat[:, :eb] = ds_mla_records(rng, nb * block_size)
    if fmt == FP8:
        q = normal_e4m3_codes(rng, (B * q_len, H, 576), 1.0 / q_scale)
    else:
        q = normal_bf16_bits(rng, (B * q_len, H, 576)).view(np.uint8).reshape(B * q_len, H, 1152)
    return PagedCase(fmt=fmt, q=q, cache=cache, block_table=bt, seq_lens=seq_lens, q_len=q_len,
                     H=H, max_context=int(max_context), softmax_scale=SOFTMAX_SCALE,
                     q_scale=q_scale, k_scale=k_scale, return_lse=return_lse,
                     meta=dict(B=B, L_lo=L_lo, L_hi=L_hi, block_size=block_size))


@dataclass
class EpilogueInputs:
    ql_nope: np.ndarray      # uint16 [B, H, 512]
    q_pe: np.ndarray         # uint16 [B, H, 64]
    kv_c: np.ndarray         # uint16 [B, 512]
    k_pe: np.ndarray         # uint16 [B, 64]
    positions: np.ndarray    # int64 [B]
    slot_mapping: np.ndarray  # int64 [B]
    cos_sin: np.ndarray      # fp32 [max_position, 64]


def epilogue_inputs(seed: int, B: int, H: int, slot_mapping, positions,
                    max_position: int = 131072) -> EpilogueInputs:
    rng = np.random.default_rng(seed + 1000)
    return EpilogueInputs(
        ql_nope=normal_bf16_bits(rng, (B, H, 512)), q_pe=normal_bf16_bits(rng, (B, H, 64)),
        kv_c=normal_bf16_bits(rng, (B, 512)), k_pe=normal_bf16_bits(rng, (B, 64)),
        positions=np.asarray(positions, dtype=np.int64),
        slot_mapping=np.asarray(slot_mapping, dtype=np.int64),
        cos_sin=cos_sin_table(max_position))


def last_token_slots(case: PagedCase) -> np.ndarray:
    """Slot of each request's last key position (where the decode token is inserted)."""
    bs = case.cache.shape[1]
    L = case.seq_lens.astype(np.int64)
    p = L - 1
    return case.block_table[np.arange(L.size), p // bs].astype(np.int64) * bs + p % bs


def config1(B: int = 32, L_lo: int = 1024, L_hi: int = 8192):
    """Paged bf16 decode + epilogue: B=32, q=1, H=16, block_size=64, seq_lens ~ U[1024, 8192],
    shuffled block table; epilogue inputs N(0,1) bf16 with positions L-1 and the slot of
    position L-1; cos/sin table max_position 131072, base 10000; seed 1."""
    case = paged_case(1, BF16, B=B, q_len=1, H=16, L_lo=L_lo, L_hi=L_hi, block_size=64,
                      max_context=L_hi)
    slots = last_token_slots(case)
    epi = epilogue_inputs(1, B, 16, slots, case.seq_lens.astype(np.int64) - 1)
    return case, epi


def config3(B: int = 64, L_lo: int = 16384, L_hi: int = 131072, max_context: int = 131072):
    """fp8 spec-verify: B=64, q=4 causal, H=16, plain fp8 cache and query with
    q_scale = k_scale = 0.05, block_size 64, L ~ U[16384, 131072], max_context 131072; seed 3."""
    return paged_case(3, FP8, B=B, q_len=4, H=16, L_lo=L_lo, L_hi=L_hi, block_size=64,
                      max_context=max_context, q_scale=0.05, k_scale=0.05)


def config4(B: int = 128, L_lo: int = 8192, L_hi: int = 32768):
    """ds_mla large-batch decode: B=128, q=1, H=96, block_size 64, unpadded 656-byte pitch,
    L ~ U[8192, 32768], bf16 query, no lse; seed 4."""
    return paged_case(4, DS_MLA, B=B, q_len=1, H=96, L_lo=L_lo, L_hi=L_hi, block_size=64,
                      max_context=L_hi, return_lse=False)


def algorithmic_bytes_sparse(case: SparseCase, H: int | None = None) -> int:
    """Records gathered (valid keys only) + q read + out written (+ lse)."""
    T = case.q.shape[0]
    H = case.q.shape[1] if H is None else H
    valid = int((case.indices >= 0).sum()) if case.has_invalid else int(case.indices.size)
    b = valid * 656 + T * H * 576 * 2 + T * H * 512 * 2
    if case.return_lse:
        b += T * H * 4
    return b


def algorithmic_bytes_paged(case: PagedCase) -> int:
    eb = ENTRY_BYTES[case.fmt]
    qe = 1 if case.fmt == FP8 else 2
    B = case.seq_lens.size
    H = case.H
    keys = int(np.maximum(case.seq_lens.astype(np.int64), 0).sum())   # each request's KV read once
    rows = B * case.q_len
    b = keys * eb + rows * H * 576 * qe + rows * H * 512 * 2
    if case.return_lse:
        b += rows * H * 4
    return b


def qk_pv_flops_paged(case: PagedCase) -> int:
    B = case.seq_lens.size
    keys = int(case.seq_lens.astype(np.int64).sum())
    return keys * case.q_len * case.H * (2 * 576 + 2 * 512)
