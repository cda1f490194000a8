/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for MLA over the 576-wide latent cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA kernels are checked
 * against.  Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
 * load it; the product path never does.  It shares no code, header, table or constant with
 * the CUDA library: every codec and formula below is written out again from its definition.
 *
 * Sources (pages on vLLM's Kimi-K3 MLA):
 *  - "vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla", flydsl_sparse_mla_fp8ds_fwd docstring:
 *    record = 512 e4m3 | 4 fp32 per-128 scales | 64 bf16 rope; CSR rows
 *    kv_indices[kv_indptr[t]:kv_indptr[t+1]]; entries < 0 masked when has_invalid;
 *    lse = natural-log log-sum-exp of softmax_scale * q.k over unmasked keys; a row with no
 *    unmasked key gives out = 0 and lse = -inf.
 *  - "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.prepared", PreparedMla and
 *    trtllm_decode: paged decode of q query tokens per request, causal among them;
 *    bmm1_scale = softmax_scale * q_scale * k_scale and bmm2_scale = k_scale for the plain
 *    fp8 cache.
 *  - "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
 *    fused_mla_decode_q_concat_kv_cache_insert: mqa_q = [ql_nope | q_pe] and insertion of
 *    [kv_c_normed | k_pe] at slot_mapping, dispatched by cache format (bf16; plain fp8 with
 *    q_scale_inv / cache_scale_inv; fp8_ds_mla with per-tile scales), optional GPT-J RoPE
 *    from an fp32 cos/sin table.
 *  - "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla", fp8_word: the fp8
 *    write is vLLM's saturating E4M3 quant.
 *  - "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
 *    fused_mla_key_concat_kv_cache_insert / fused_mla_key_concat_ds_mla_insert (prefill: full
 *    key [k_nope | k_pe] per head, q RoPE in place, latent insert) and
 *    fused_mla_qkv_quant_kv_cache_fp8_insert (fp8 q / k / v with separate scales, cache with
 *    its own scale).
 *  - "vllm.models.kimi_k3.nvidia.mla", _attention / _v_up_proj / forward: BMM1 of the decode
 *    query with W_UK_T, the W_UV up-projection of the latent output, the sigmoid output gate.
 *  - "vllm.models.kimi_k3.nvidia.mla", _compute_prefill_context / _gather_context_latent (the
 *    chunked context gathered from the paged cache into a dense workspace, up-converted or as
 *    stored) and _forward_prefill_fused (merge_attn_states of prefix and suffix partials).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - fp8_ds_mla tile scale on insert: s = 2^k with k the smallest integer such that
 *    amax <= 448 * 2^k (k clamped to >= -126), s = 1 when amax == 0; code = e4m3(x / s).
 *  - E4M3 saturating quant: clamp |x| to 448, round to nearest even on the E4M3 grid
 *    (subnormals included), NaN -> 0x7F, sign kept.
 *  - cos/sin table row p: columns 0..31 cos(p*theta_i), 32..63 sin(p*theta_i); GPT-J pairs
 *    (2i, 2i+1): y0 = fma(x0, c, -(x1*s)), y1 = fma(x1, c, x0*s), fp32 arithmetic.
 *  - spec-verify: seq_lens count the q new tokens; query row i of a request of length L
 *    sees key positions 0 .. L-q+i.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fused multiply-adds except
 * the explicit fmaf calls of the RoPE contract).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KV_LORA 512
#define ROPE 64
#define ENTRY 576

enum { ORC_BF16 = 0, ORC_FP8 = 1, ORC_DS_MLA = 2 };

/* ------------------------------------------------------------------------------------ */
/* Codecs, from the number formats' definitions.                                        */
/* ------------------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, largest finite magnitude 448. */
double orc_e4m3_to_double(uint8_t b) {
  int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);           /* subnormal: m/8 * 2^(1-7) */
  else
    v = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* Saturating round-to-nearest-even into E4M3, by brute force over the 127 non-negative
 * finite codes (they are ordered by value).  Ties go to the even code. */
uint8_t orc_e4m3_from_float_sat(float xf) {
  double x = (double)xf, a;
  int neg, c, best = 0;
  double bestd = INFINITY;
  if (isnan(x)) return 0x7F;
  neg = signbit(x) ? 1 : 0;
  a = fabs(x);
  if (a > 448.0) a = 448.0;
  for (c = 0; c <= 0x7E; ++c) {
    double d = fabs(orc_e4m3_to_double((uint8_t)c) - a);
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      bestd = d;
      best = c;
    }
  }
  return (uint8_t)(best | (neg << 7));
}

/* bfloat16: the top half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* binary32 -> bfloat16, round to nearest even; NaN becomes the quiet NaN 0x7FC0 (sign kept). */
uint16_t orc_bf16_from_float(float f) {
  uint32_t u, lsb;
  memcpy(&u, &f, 4);
  if (isnan(f)) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
  lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static float bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFF);
  p[1] = (uint8_t)(v >> 8);
}
static float rdf32(const uint8_t* p) {
  float f;
  memcpy(&f, p, 4); /* both hosts are little-endian, as is the device */
  return f;
}

/* ------------------------------------------------------------------------------------ */
/* Cache entry decode.                                                                   */
/* ------------------------------------------------------------------------------------ */

/* One cache entry -> 576 exact values.  fp8_ds_mla: NoPE d < 512 is e4m3(b[d]) times the
 * fp32 scale of its 128-wide tile (bytes 512 + 4*(d/128)); rope is the bf16 at bytes
 * 528 + 2i.  Plain fp8: all 576 are e4m3 (the per-tensor k_scale is applied by the
 * caller).  bf16: 576 little-endian bf16 values. */
void orc_decode_entry(int fmt, const uint8_t* e, double* k) {
  int d;
  if (fmt == ORC_BF16) {
    for (d = 0; d < ENTRY; ++d) k[d] = orc_bf16_to_double(rd16(e + 2 * d));
  } else if (fmt == ORC_FP8) {
    for (d = 0; d < ENTRY; ++d) k[d] = orc_e4m3_to_double(e[d]);
  } else {
    double s[4];
    for (d = 0; d < 4; ++d) s[d] = (double)rdf32(e + KV_LORA + 4 * d);
    for (d = 0; d < KV_LORA; ++d) k[d] = orc_e4m3_to_double(e[d]) * s[d / 128];
    for (d = 0; d < ROPE; ++d) k[KV_LORA + d] = orc_bf16_to_double(rd16(e + KV_LORA + 16 + 2 * d));
  }
}

/* ------------------------------------------------------------------------------------ */
/* Attention of one query vector over a key set (plain two-pass definition).            */
/* ------------------------------------------------------------------------------------ */

/* x_k = sigma * sum_d q[d] K_k[d];  lse = ln sum_k exp(x_k);
 * out[d] = out_scale * sum_k exp(x_k - lse) * K_k[d] for d < 512.
 * n == 0: out = 0, lse = -inf. */
static void attend_one(const double* qv, const double* K, int64_t n, double sigma,
                       double out_scale, double* x, double* out, double* lse) {
  int64_t k;
  int d;
  double m = -INFINITY, l = 0.0, ls;
  for (d = 0; d < KV_LORA; ++d) out[d] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  for (k = 0; k < n; ++k) {
    const double* kv = K + k * ENTRY;
    double acc = 0.0;
    for (d = 0; d < ENTRY; ++d) acc += qv[d] * kv[d];
    x[k] = sigma * acc;
    if (x[k] > m) m = x[k];
  }
  for (k = 0; k < n; ++k) l += exp(x[k] - m);
  ls = m + log(l);
  for (k = 0; k < n; ++k) {
    const double* kv = K + k * ENTRY;
    double w = exp(x[k] - ls);
    for (d = 0; d < KV_LORA; ++d) out[d] += w * kv[d];
  }
  for (d = 0; d < KV_LORA; ++d) out[d] *= out_scale;
  *lse = ls;
}

/* ------------------------------------------------------------------------------------ */
/* Sparse forward over fp8_ds_mla records (CSR key lists).                               */
/* ------------------------------------------------------------------------------------ */

/* q: bf16 [T, H, 576] with element strides q_s0 / q_s1 (unit last stride).
 * records: num_records entries of 656 bytes at record_stride bytes.
 * indptr [T+1], indices [indptr[T]] (int64 here; the test harness widens).
 * rows: optional list of n_rows query rows to compute (NULL = all T, in order).
 * out: [n_rows, H, 512] fp64; lse: [n_rows, H] fp64.
 * Returns 0, or -1 when an index is out of range and not a masked negative. */
int orc_sparse_fwd(const uint16_t* q, int64_t q_s0, int64_t q_s1, const uint8_t* records,
                   int64_t record_stride, int64_t num_records, const int64_t* indptr,
                   const int64_t* indices, double softmax_scale, int has_invalid, int T, int H,
                   const int32_t* rows, int n_rows, double* out, double* lse) {
  int bad = 0;
  int ri;
  if (rows == NULL) n_rows = T;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (ri = 0; ri < n_rows; ++ri) {
    int t = rows ? rows[ri] : ri;
    int64_t b = indptr[t], e = indptr[t + 1], j, n = 0;
    double* K = (double*)malloc(sizeof(double) * ENTRY * (size_t)((e - b) > 0 ? (e - b) : 1));
    double* x = (double*)malloc(sizeof(double) * (size_t)((e - b) > 0 ? (e - b) : 1));
    double qv[ENTRY];
    int h, d;
    for (j = b; j < e; ++j) {
      int64_t idx = indices[j];
      if (idx < 0 && has_invalid) continue;
      if (idx < 0 || idx >= num_records) {
        bad = 1;
        continue;
      }
      orc_decode_entry(ORC_DS_MLA, records + idx * record_stride, K + n * ENTRY);
      ++n;
    }
    for (h = 0; h < H; ++h) {
      const uint16_t* qp = q + (int64_t)t * q_s0 + (int64_t)h * q_s1;
      for (d = 0; d < ENTRY; ++d) qv[d] = orc_bf16_to_double(qp[d]);
      attend_one(qv, K, n, softmax_scale, 1.0, x, out + ((int64_t)ri * H + h) * KV_LORA,
                 lse + (int64_t)ri * H + h);
    }
    free(K);
    free(x);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* Sparse forward with the general op's extras: attention sink and a second KV segment.  */
/* ------------------------------------------------------------------------------------ */

/* "vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla", flydsl_sparse_mla_fp8ds_supported: the
 * general sparse_mla_fwd also takes attn_sink, a second key segment (extra_kv, extra_indptr,
 * extra_indices) and kv_splits, which the FlyDSL slice refuses.  The page names them only;
 * the readings taken here:
 *   - extra segment: row t attends the union (a multiset) of its keys in the first segment
 *     (kv_indices[kv_indptr[t]..] into records) and in the second (extra_indices
 *     [extra_indptr[t]..] into extra_records), under one softmax; negative entries of either
 *     are masked when has_invalid;
 *   - attn_sink[h]: a logit of head h (natural-log units, like softmax_scale * q.k) that
 *     joins the softmax denominator with a zero value:
 *       lse = ln(sum_k e^{x_k} + e^{sink_h}),  out = sum_k e^{x_k - lse} V_k,
 *     so a row without keys gives out = 0 and lse = sink_h (sink = -inf: no sink);
 *   - kv_splits: a partition of each row's key list for parallelism, which leaves the
 *     result unchanged (this function has no counterpart of it).
 * Arguments as orc_sparse_fwd, plus records2 / indptr2 / indices2 (all NULL: no second
 * segment) and sink [H] (NULL: none). */
int orc_sparse_fwd_ext(const uint16_t* q, int64_t q_s0, int64_t q_s1, const uint8_t* records,
                       int64_t record_stride, int64_t num_records, const int64_t* indptr, const int64_t* indices,
                       const uint8_t* records2, int64_t record_stride2, int64_t num_records2,
                       const int64_t* indptr2, const int64_t* indices2, const float* sink, double softmax_scale,
                       int has_invalid, int T, int H, double* out, double* lse) {
  int bad = 0;
  int t;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (t = 0; t < T; ++t) {
    int64_t n1 = indptr[t + 1] - indptr[t], n2 = records2 ? indptr2[t + 1] - indptr2[t] : 0, j, n = 0;
    int64_t cap = (n1 > 0 ? n1 : 0) + (n2 > 0 ? n2 : 0);
    double* K = (double*)malloc(sizeof(double) * ENTRY * (size_t)(cap > 0 ? cap : 1));
    double* x = (double*)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
    double qv[ENTRY];
    int h, d, seg;
    for (seg = 0; seg < 2; ++seg) {
      const uint8_t* rec = seg ? records2 : records;
      int64_t stride = seg ? record_stride2 : record_stride, nrec = seg ? num_records2 : num_records;
      const int64_t* ptr = seg ? indptr2 : indptr;
      const int64_t* idxs = seg ? indices2 : indices;
      if (!rec) continue;
      for (j = ptr[t]; j < ptr[t + 1]; ++j) {
        int64_t idx = idxs[j];
        if (idx < 0 && has_invalid) continue;
        if (idx < 0 || idx >= nrec) {
          bad = 1;
          continue;
        }
        orc_decode_entry(ORC_DS_MLA, rec + idx * stride, K + n * ENTRY);
        ++n;
      }
    }
    for (h = 0; h < H; ++h) {
      const uint16_t* qp = q + (int64_t)t * q_s0 + (int64_t)h * q_s1;
      double* o = out + ((int64_t)t * H + h) * KV_LORA;
      double sk = sink ? (double)sink[h] : -INFINITY, m = sk, l = 0.0, ls;
      int64_t k;
      for (d = 0; d < ENTRY; ++d) qv[d] = orc_bf16_to_double(qp[d]);
      for (d = 0; d < KV_LORA; ++d) o[d] = 0.0;
      for (k = 0; k < n; ++k) {
        double acc = 0.0;
        for (d = 0; d < ENTRY; ++d) acc += qv[d] * K[k * ENTRY + d];
        x[k] = softmax_scale * acc;
        if (x[k] > m) m = x[k];
      }
      if (m == -INFINITY) {
        lse[(int64_t)t * H + h] = -INFINITY;
        continue;
      }
      for (k = 0; k < n; ++k) l += exp(x[k] - m);
      if (sk > -INFINITY) l += exp(sk - m);
      ls = m + log(l);
      for (k = 0; k < n; ++k) {
        double w = exp(x[k] - ls);
        for (d = 0; d < KV_LORA; ++d) o[d] += w * K[k * ENTRY + d];
      }
      lse[(int64_t)t * H + h] = ls;
    }
    free(K);
    free(x);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* Paged decode / spec-verify.                                                           */
/* ------------------------------------------------------------------------------------ */

/* q: [B*q_len, H, 576], bf16 (formats bf16, ds_mla) or e4m3 bytes (plain fp8); byte
 * strides q_s0_bytes / q_s1_bytes.  Request b's key positions are 0 .. L_b-1 with
 * L_b = seq_lens[b]; query row i (0 <= i < q_len) sees positions 0 .. L_b - q_len + i.
 * Position p lives at block block_table[b*bt_stride + p/block_size], offset p%block_size:
 * entry address = cache + block*block_stride + (p%block_size)*entry_stride (bytes).
 * sigma = softmax_scale (bf16, ds_mla) or softmax_scale*q_scale*k_scale (plain fp8, with
 * q and K the raw e4m3 values); the fp8 output is multiplied by k_scale.
 * rows: optional list of query rows (b*q_len + i); NULL = all.
 * Returns 0, or -1 if a block id is out of [0, num_blocks). */
int orc_paged_decode(int fmt, const uint8_t* q, int64_t q_s0_bytes, int64_t q_s1_bytes,
                     const uint8_t* cache, int64_t num_blocks, int64_t block_stride,
                     int64_t entry_stride, int block_size, const int32_t* block_table,
                     int64_t bt_stride, const int32_t* seq_lens, int B, int q_len, int H,
                     double softmax_scale, double q_scale, double k_scale, const int32_t* rows,
                     int n_rows, double* out, double* lse) {
  int bad = 0;
  int ri;
  double sigma = softmax_scale, oscale = 1.0;
  if (fmt == ORC_FP8) {
    sigma = softmax_scale * q_scale * k_scale;
    oscale = k_scale;
  }
  if (rows == NULL) n_rows = B * q_len;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (ri = 0; ri < n_rows; ++ri) {
    int row = rows ? rows[ri] : ri;
    int b = row / q_len, i = row % q_len;
    int64_t L = seq_lens[b];
    int64_t n = L - q_len + i + 1, p, nn = 0;
    double *K, *x, qv[ENTRY];
    int h, d;
    if (n < 0) n = 0;
    K = (double*)malloc(sizeof(double) * ENTRY * (size_t)(n > 0 ? n : 1));
    x = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (p = 0; p < n; ++p) {
      int64_t blk = block_table[(int64_t)b * bt_stride + p / block_size];
      if (blk < 0 || blk >= num_blocks) {
        bad = 1;
        continue;
      }
      orc_decode_entry(fmt, cache + blk * block_stride + (p % block_size) * entry_stride,
                       K + nn * ENTRY);
      ++nn;
    }
    for (h = 0; h < H; ++h) {
      const uint8_t* qp = q + (int64_t)row * q_s0_bytes + (int64_t)h * q_s1_bytes;
      for (d = 0; d < ENTRY; ++d)
        qv[d] = (fmt == ORC_FP8) ? orc_e4m3_to_double(qp[d]) : orc_bf16_to_double(rd16(qp + 2 * d));
      attend_one(qv, K, nn, sigma, oscale, x, out + ((int64_t)ri * H + h) * KV_LORA,
                 lse + (int64_t)ri * H + h);
    }
    free(K);
    free(x);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* Merge of partial attentions by their log-sum-exp (the chunk / split combine).         */
/* ------------------------------------------------------------------------------------ */

/* parts: S partial outputs of width 512 (each normalised by its own sum), lse_parts: S.
 * lse = ln sum_s exp(lse_s); out = sum_s exp(lse_s - lse) * parts_s.  All -inf -> 0, -inf. */
void orc_merge(int S, const double* parts, const double* lse_parts, double* out, double* lse) {
  double m = -INFINITY, l = 0.0;
  int s, d;
  for (d = 0; d < KV_LORA; ++d) out[d] = 0.0;
  for (s = 0; s < S; ++s)
    if (lse_parts[s] > m) m = lse_parts[s];
  if (m == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  for (s = 0; s < S; ++s) l += exp(lse_parts[s] - m);
  *lse = m + log(l);
  for (s = 0; s < S; ++s) {
    double w = exp(lse_parts[s] - *lse);
    for (d = 0; d < KV_LORA; ++d) out[d] += w * parts[(int64_t)s * KV_LORA + d];
  }
}

/* ------------------------------------------------------------------------------------ */
/* Decode epilogue: q concat + latent insert.                                            */
/* ------------------------------------------------------------------------------------ */

/* GPT-J rotation of one 64-wide vector in fp32 (the epilogue's RoPE contract). */
static void rope_fp32(const float* x, const float* cs_row, float* y) {
  int i;
  for (i = 0; i < ROPE / 2; ++i) {
    float c = cs_row[i], s = cs_row[ROPE / 2 + i];
    float x0 = x[2 * i], x1 = x[2 * i + 1];
    float t0 = x1 * s; /* rounded fp32 product (no contraction in this file) */
    float t1 = x0 * s;
    y[2 * i] = fmaf(x0, c, -t0);
    y[2 * i + 1] = fmaf(x1, c, t1);
  }
}

/* Smallest integer k with amax <= 448 * 2^k, clamped to k >= -126; amax == 0 -> k = 0. */
static int ds_tile_exponent(double amax) {
  int e, k;
  double f;
  if (amax == 0.0) return 0;
  f = frexp(amax, &e); /* amax = f * 2^e, 0.5 <= f < 1; 448 = 0.875 * 2^9 */
  k = e - 9 + (f > 0.875 ? 1 : 0);
  if (k < -126) k = -126;
  return k;
}

/* Write one cache entry from the latent kc (512 bf16 values) and the rotated rope kpr (64
 * fp32 values): bf16 [kc | bf16(kpr)]; plain fp8 e4m3_sat(x * cache_scale_inv) for all 576;
 * fp8_ds_mla per-128-tile power-of-two scale s_j (ds_tile_exponent of the tile's amax),
 * codes e4m3_sat(x / s_j), the four scales as fp32 at byte 512, bf16(kpr) at byte 528. */
static void write_latent(int fmt, uint8_t* ent, const uint16_t* kc, const float* kpr, float cache_scale_inv) {
  float x[KV_LORA];
  int d;
  for (d = 0; d < KV_LORA; ++d) x[d] = bf16_to_float(kc[d]);
  if (fmt == ORC_BF16) {
    for (d = 0; d < KV_LORA; ++d) wr16(ent + 2 * d, kc[d]);
    for (d = 0; d < ROPE; ++d) wr16(ent + 2 * (KV_LORA + d), orc_bf16_from_float(kpr[d]));
  } else if (fmt == ORC_FP8) {
    for (d = 0; d < KV_LORA; ++d) ent[d] = orc_e4m3_from_float_sat(x[d] * cache_scale_inv);
    for (d = 0; d < ROPE; ++d) ent[KV_LORA + d] = orc_e4m3_from_float_sat(kpr[d] * cache_scale_inv);
  } else {
    int j;
    for (j = 0; j < 4; ++j) {
      double amax = 0.0, s;
      float sf;
      int k;
      for (d = 0; d < 128; ++d) {
        double a = fabs((double)x[128 * j + d]);
        if (a > amax) amax = a;
      }
      k = ds_tile_exponent(amax);
      s = ldexp(1.0, k);
      sf = (float)s;
      memcpy(ent + KV_LORA + 4 * j, &sf, 4);
      for (d = 0; d < 128; ++d)
        ent[128 * j + d] = orc_e4m3_from_float_sat((float)((double)x[128 * j + d] / s));
    }
    for (d = 0; d < ROPE; ++d) wr16(ent + KV_LORA + 16 + 2 * d, orc_bf16_from_float(kpr[d]));
  }
}

/* Inputs are bf16 tensors given by element strides (unit last stride):
 *   ql_nope [B, H, 512], q_pe [B, H, 64], kv_c [B, 512], k_pe [B, 64].
 * mqa_q out: [B, H, 576] contiguous, bf16 (bf16 / ds_mla formats) or e4m3 bytes (plain fp8).
 * cache: num_blocks blocks at block_stride bytes, entries at entry_stride bytes.
 * slot_mapping [B] int64, < 0 skips the insert (mqa_q is still written); a slot whose
 * block is out of range is skipped too and reported by the return value -1.
 * positions [B] int64 and cos_sin [max_position, 64] fp32: both NULL (no RoPE) or both set.
 * q_scale_inv / cache_scale_inv: used by the plain fp8 format only. */
int orc_q_concat_cache_insert(int fmt, const uint16_t* ql_nope, int64_t ql_s0, int64_t ql_s1,
                              const uint16_t* q_pe, int64_t qp_s0, int64_t qp_s1,
                              const uint16_t* kv_c, int64_t kv_s0, const uint16_t* k_pe,
                              int64_t kp_s0, uint8_t* mqa_q, uint8_t* cache, int64_t num_blocks,
                              int64_t block_stride, int64_t entry_stride, int block_size,
                              const int64_t* slot_mapping, float q_scale_inv,
                              float cache_scale_inv, const int64_t* positions,
                              const float* cos_sin, int64_t max_position, int B, int H) {
  int bad = 0, b;
  for (b = 0; b < B; ++b) {
    const float* cs = NULL;
    float kp[ROPE], kpr[ROPE];
    int h, d;
    int64_t slot;
    if (positions) {
      int64_t pos = positions[b];
      if (pos < 0 || pos >= max_position) {
        bad = 1;
        pos = pos < 0 ? 0 : max_position - 1;
      }
      cs = cos_sin + pos * ROPE;
    }
    /* query concat */
    for (h = 0; h < H; ++h) {
      const uint16_t* qn = ql_nope + (int64_t)b * ql_s0 + (int64_t)h * ql_s1;
      const uint16_t* qp = q_pe + (int64_t)b * qp_s0 + (int64_t)h * qp_s1;
      float qpf[ROPE], qpr[ROPE];
      uint8_t* dst = mqa_q + ((int64_t)b * H + h) * ENTRY * (fmt == ORC_FP8 ? 1 : 2);
      for (d = 0; d < ROPE; ++d) qpf[d] = bf16_to_float(qp[d]);
      if (cs)
        rope_fp32(qpf, cs, qpr);
      else
        memcpy(qpr, qpf, sizeof qpr);
      if (fmt == ORC_FP8) {
        for (d = 0; d < KV_LORA; ++d) dst[d] = orc_e4m3_from_float_sat(bf16_to_float(qn[d]) * q_scale_inv);
        for (d = 0; d < ROPE; ++d) dst[KV_LORA + d] = orc_e4m3_from_float_sat(qpr[d] * q_scale_inv);
      } else {
        for (d = 0; d < KV_LORA; ++d) wr16(dst + 2 * d, qn[d]);
        for (d = 0; d < ROPE; ++d) wr16(dst + 2 * (KV_LORA + d), orc_bf16_from_float(qpr[d]));
      }
    }
    /* latent insert */
    slot = slot_mapping[b];
    if (slot < 0) continue;
    if (slot / block_size >= num_blocks) {
      bad = 1;
      continue;
    }
    {
      uint8_t* ent = cache + (slot / block_size) * block_stride + (slot % block_size) * entry_stride;
      const uint16_t* kr = k_pe + (int64_t)b * kp_s0;
      for (d = 0; d < ROPE; ++d) kp[d] = bf16_to_float(kr[d]);
      if (cs)
        rope_fp32(kp, cs, kpr);
      else
        memcpy(kpr, kp, sizeof kpr);
      write_latent(fmt, ent, kv_c + (int64_t)b * kv_s0, kpr, cache_scale_inv);
    }
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* Prefill epilogues: full-key concat, in-place query RoPE, latent insert, fp8 q/k/v quant. */
/* ------------------------------------------------------------------------------------ */

/* The RoPE row of token t (NULL without RoPE); an out-of-range position is clamped and
 * reported through *bad. */
static const float* rope_row(const int64_t* positions, const float* cos_sin, int64_t max_position, int t,
                             int* bad) {
  int64_t pos;
  if (!positions) return NULL;
  pos = positions[t];
  if (pos < 0 || pos >= max_position) {
    *bad = 1;
    pos = pos < 0 ? 0 : max_position - 1;
  }
  return cos_sin + pos * ROPE;
}

/* bf16 vector of 64 -> rotated fp32 (or the plain values without RoPE). */
static void rope_bf16_vec(const uint16_t* x, const float* cs, float* y) {
  float xf[ROPE];
  int d;
  for (d = 0; d < ROPE; ++d) xf[d] = bf16_to_float(x[d]);
  if (cs)
    rope_fp32(xf, cs, y);
  else
    memcpy(y, xf, sizeof xf);
}

/* "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
 * fused_mla_key_concat_kv_cache_insert (fmt = bf16) and fused_mla_key_concat_ds_mla_insert
 * (fmt = fp8_ds_mla).  Per prefill token t (Tp tokens), H heads, dn NoPE dims per head:
 *   q      bf16 [Tp, H, dn + 64] (element strides q_s0, q_s1): its last 64 values are
 *          rotated in place when positions are given (bf16 of the fp32 rotation);
 *   k_nope bf16 [Tp, H, dn]; k_pe bf16 [Tp, 64]; kv_c bf16 [Tp, 512];
 *   k_out  bf16 [Tp, H, dn + 64] contiguous: [k_nope[t, h] | bf16(rope(k_pe[t]))];
 *   the latent [kv_c | rope(k_pe)] is written at slot_mapping[t] as in the decode epilogue
 *   (a negative slot skips it).
 * Returns -1 if a slot's block or a position is out of range (skipped / clamped). */
int orc_key_concat_cache_insert(int fmt, uint16_t* q, int64_t q_s0, int64_t q_s1, const uint16_t* k_nope,
                                int64_t kn_s0, int64_t kn_s1, const uint16_t* k_pe, int64_t kp_s0,
                                const uint16_t* kv_c, int64_t kv_s0, uint16_t* k_out, uint8_t* cache,
                                int64_t num_blocks, int64_t block_stride, int64_t entry_stride, int block_size,
                                const int64_t* slot_mapping, const int64_t* positions, const float* cos_sin,
                                int64_t max_position, int Tp, int H, int dn) {
  int bad = 0, t, h, d;
  for (t = 0; t < Tp; ++t) {
    const float* cs = rope_row(positions, cos_sin, max_position, t, &bad);
    float kpr[ROPE];
    int64_t slot;
    rope_bf16_vec(k_pe + (int64_t)t * kp_s0, cs, kpr);
    for (h = 0; h < H; ++h) {
      uint16_t* qh = q + (int64_t)t * q_s0 + (int64_t)h * q_s1;
      const uint16_t* kn = k_nope + (int64_t)t * kn_s0 + (int64_t)h * kn_s1;
      uint16_t* ko = k_out + ((int64_t)t * H + h) * (dn + ROPE);
      if (cs) {
        float qr[ROPE];
        rope_bf16_vec(qh + dn, cs, qr);
        for (d = 0; d < ROPE; ++d) qh[dn + d] = orc_bf16_from_float(qr[d]);
      }
      for (d = 0; d < dn; ++d) ko[d] = kn[d];
      for (d = 0; d < ROPE; ++d) ko[dn + d] = orc_bf16_from_float(kpr[d]);
    }
    slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot / block_size >= num_blocks) {
      bad = 1;
      continue;
    }
    write_latent(fmt, cache + (slot / block_size) * block_stride + (slot % block_size) * entry_stride,
                 kv_c + (int64_t)t * kv_s0, kpr, 1.0f);
  }
  return bad ? -1 : 0;
}

/* "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
 * fused_mla_qkv_quant_kv_cache_fp8_insert.  Per token t and head h (dn NoPE dims, dv value
 * dims), with x -> e4m3_sat(x * inv) the saturating quant of the fp32 product:
 *   q_fp8 [Tp, H, dn + 64] = quant([q_nope | rope(q_pe)], q_scale_inv)   (q is not modified);
 *   k_fp8 [Tp, H, dn + 64] = quant([k_nope | rope(k_pe)], k_scale_inv);
 *   v_fp8 [Tp, H, dv]      = quant(v, v_scale_inv);
 *   cache entry at slot    = quant([kv_c | rope(k_pe)], cache_scale_inv) (plain fp8 cache).
 * Outputs are contiguous; inputs use element strides.  Returns -1 as above. */
int orc_qkv_quant_cache_fp8_insert(const uint16_t* q, int64_t q_s0, int64_t q_s1, const uint16_t* k_nope,
                                   int64_t kn_s0, int64_t kn_s1, const uint16_t* k_pe, int64_t kp_s0,
                                   const uint16_t* kv_c, int64_t kv_s0, const uint16_t* v, int64_t v_s0,
                                   int64_t v_s1, uint8_t* q_fp8, uint8_t* k_fp8, uint8_t* v_fp8, uint8_t* cache,
                                   int64_t num_blocks, int64_t block_stride, int64_t entry_stride, int block_size,
                                   const int64_t* slot_mapping, float q_scale_inv, float k_scale_inv,
                                   float v_scale_inv, float cache_scale_inv, const int64_t* positions,
                                   const float* cos_sin, int64_t max_position, int Tp, int H, int dn, int dv) {
  int bad = 0, t, h, d;
  for (t = 0; t < Tp; ++t) {
    const float* cs = rope_row(positions, cos_sin, max_position, t, &bad);
    float kpr[ROPE];
    int64_t slot;
    rope_bf16_vec(k_pe + (int64_t)t * kp_s0, cs, kpr);
    for (h = 0; h < H; ++h) {
      const uint16_t* qh = q + (int64_t)t * q_s0 + (int64_t)h * q_s1;
      const uint16_t* kn = k_nope + (int64_t)t * kn_s0 + (int64_t)h * kn_s1;
      const uint16_t* vh = v + (int64_t)t * v_s0 + (int64_t)h * v_s1;
      uint8_t* qo = q_fp8 + ((int64_t)t * H + h) * (dn + ROPE);
      uint8_t* ko = k_fp8 + ((int64_t)t * H + h) * (dn + ROPE);
      uint8_t* vo = v_fp8 + ((int64_t)t * H + h) * dv;
      float qr[ROPE];
      rope_bf16_vec(qh + dn, cs, qr);
      for (d = 0; d < dn; ++d) qo[d] = orc_e4m3_from_float_sat(bf16_to_float(qh[d]) * q_scale_inv);
      for (d = 0; d < ROPE; ++d) qo[dn + d] = orc_e4m3_from_float_sat(qr[d] * q_scale_inv);
      for (d = 0; d < dn; ++d) ko[d] = orc_e4m3_from_float_sat(bf16_to_float(kn[d]) * k_scale_inv);
      for (d = 0; d < ROPE; ++d) ko[dn + d] = orc_e4m3_from_float_sat(kpr[d] * k_scale_inv);
      for (d = 0; d < dv; ++d) vo[d] = orc_e4m3_from_float_sat(bf16_to_float(vh[d]) * v_scale_inv);
    }
    slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot / block_size >= num_blocks) {
      bad = 1;
      continue;
    }
    write_latent(ORC_FP8, cache + (slot / block_size) * block_stride + (slot % block_size) * entry_stride,
                 kv_c + (int64_t)t * kv_s0, kpr, cache_scale_inv);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* Chunked-context prefill: gather of the paged context, and the prefix / suffix merge.   */
/* ------------------------------------------------------------------------------------ */

/* "vllm.models.kimi_k3.nvidia.mla", _gather_context_latent (cp_gather_and_upconvert_fp8_kv_cache
 * for fp8_ds_mla, gather_and_maybe_dequant_cache for bf16 / plain fp8 with a bf16 query,
 * cp_gather_cache for plain fp8 with an fp8 query).  Request b of the chunk (batch requests)
 * owns output rows cu_seq_lens[b] .. cu_seq_lens[b+1]-1; row cu_seq_lens[b] + i holds context
 * position p = seq_starts[b] + i (seq_starts NULL: 0) of request b, found through
 * block_table[b * bt_stride + p / block_size] at offset p % block_size.
 *   out_kind 0: dst rows of 576 bf16 values (uint16 bits, dst_row elements apart): the entry's
 *     values, each dequantised in fp32 (e4m3 value times the tile scale for fp8_ds_mla, times
 *     `scale` for plain fp8; bf16 entries as stored) and rounded once to bf16;
 *   out_kind 1: dst rows of the entry's stored bytes (entry_bytes of the format, dst_row bytes
 *     apart).
 * Rows at or past cu_seq_lens[batch] (up to num_tokens) are not written.  A row whose block
 * id is out of range is written as zeros and reported by the return value -1. */
int orc_gather_context(int fmt, const uint8_t* cache, int64_t num_blocks, int64_t block_stride,
                       int64_t entry_stride, int block_size, const int32_t* block_table, int64_t bt_stride,
                       const int32_t* cu_seq_lens, const int32_t* seq_starts, int batch, int64_t num_tokens,
                       int out_kind, float scale, uint8_t* dst, int64_t dst_row) {
  int bad = 0, b, d;
  const int eb = fmt == ORC_BF16 ? 1152 : fmt == ORC_FP8 ? ENTRY : 656;
  for (b = 0; b < batch; ++b) {
    int64_t r;
    for (r = cu_seq_lens[b]; r < cu_seq_lens[b + 1] && r < num_tokens; ++r) {
      int64_t p = (seq_starts ? seq_starts[b] : 0) + (r - cu_seq_lens[b]);
      int64_t blk = block_table[(int64_t)b * bt_stride + p / block_size];
      const uint8_t* ent;
      if (out_kind == 1) {
        uint8_t* o = dst + r * dst_row;
        if (blk < 0 || blk >= num_blocks) {
          bad = 1;
          memset(o, 0, (size_t)eb);
          continue;
        }
        ent = cache + blk * block_stride + (p % block_size) * entry_stride;
        memcpy(o, ent, (size_t)eb);
      } else {
        uint16_t* o = (uint16_t*)(dst) + r * dst_row;
        if (blk < 0 || blk >= num_blocks) {
          bad = 1;
          for (d = 0; d < ENTRY; ++d) o[d] = 0;
          continue;
        }
        ent = cache + blk * block_stride + (p % block_size) * entry_stride;
        if (fmt == ORC_BF16) {
          for (d = 0; d < ENTRY; ++d) o[d] = rd16(ent + 2 * d);
        } else if (fmt == ORC_FP8) {
          for (d = 0; d < ENTRY; ++d) o[d] = orc_bf16_from_float((float)orc_e4m3_to_double(ent[d]) * scale);
        } else {
          for (d = 0; d < KV_LORA; ++d)
            o[d] = orc_bf16_from_float((float)orc_e4m3_to_double(ent[d]) * rdf32(ent + KV_LORA + 4 * (d / 128)));
          for (d = 0; d < ROPE; ++d) o[KV_LORA + d] = rd16(ent + KV_LORA + 16 + 2 * d);
        }
      }
    }
  }
  return bad ? -1 : 0;
}

/* "vllm.models.kimi_k3.nvidia.mla", _forward_prefill_fused: merge_attn_states of the
 * context (prefix) and new-token (suffix) partial attentions.  For token t and head h:
 *   lse = ln(e^{lse_p} + e^{lse_s}),  out = e^{lse_p - lse} O_p + e^{lse_s - lse} O_s
 * (orc_merge with two parts).  O_p, O_s: bf16 [T, H, D] with element strides; lse_p, lse_s:
 * fp32 [H, T]; out: fp64 [T, H, D]; out_lse: fp64 [H, T]. */
void orc_merge_attn_states(const uint16_t* prefix, int64_t p_s0, int64_t p_s1, const float* prefix_lse,
                           const uint16_t* suffix, int64_t s_s0, int64_t s_s1, const float* suffix_lse, int T, int H,
                           int D, double* out, double* out_lse) {
  int t, h, d;
  double* parts = (double*)malloc(sizeof(double) * 2 * KV_LORA);
  for (t = 0; t < T; ++t)
    for (h = 0; h < H; ++h) {
      double lp[2], o[KV_LORA], l;
      const uint16_t* a = prefix + (int64_t)t * p_s0 + (int64_t)h * p_s1;
      const uint16_t* c = suffix + (int64_t)t * s_s0 + (int64_t)h * s_s1;
      for (d = 0; d < KV_LORA; ++d) {
        parts[d] = d < D ? orc_bf16_to_double(a[d]) : 0.0;
        parts[KV_LORA + d] = d < D ? orc_bf16_to_double(c[d]) : 0.0;
      }
      lp[0] = (double)prefix_lse[(int64_t)h * T + t];
      lp[1] = (double)suffix_lse[(int64_t)h * T + t];
      orc_merge(2, parts, lp, o, &l);
      for (d = 0; d < D; ++d) out[((int64_t)t * H + h) * D + d] = o[d];
      out_lse[(int64_t)h * T + t] = l;
    }
  free(parts);
}

/* ------------------------------------------------------------------------------------ */
/* Absorbed decode around the attention core: the query into latent space (BMM1 with    */
/* W_UK_T) and the latent output back to the value space (W_UV), with the output gate.   */
/* ------------------------------------------------------------------------------------ */

/* "vllm.models.kimi_k3.nvidia.mla", _attention (BMM1: ql_nope = q_nope x W_UK_T per head)
 * and _v_up_proj (out = latent x W_UV per head): for token b and head h,
 *   y[b, h, f] = sum_k x[b, h, k] * w[h, k, f]
 * with x bf16 [B, H, K] (element strides x_s0, x_s1), w bf16 [H, K, F] contiguous, y fp64
 * [B, H, F], computed exactly in fp64.  When g is given (the output gate of forward,
 * _gate_sigmoid_mul, g bf16 [B, H * F] with row stride g_s0) the result is multiplied by
 * sigmoid(g[b, h * F + f]) in fp64; the rounding steps of the bf16 pipeline (the product to
 * bf16, the gate bf16(sigmoid(g)), the gated value to bf16) are left to the comparison's
 * tolerance. */
void orc_head_bmm(const uint16_t* x, int64_t x_s0, int64_t x_s1, const uint16_t* w, const uint16_t* g, int64_t g_s0,
                  int B, int H, int K, int F, double* y) {
  int b;
#pragma omp parallel for schedule(static)
  for (b = 0; b < B; ++b) {
    int h, k, f;
    double* acc = (double*)malloc(sizeof(double) * (size_t)F);
    for (h = 0; h < H; ++h) {
      const uint16_t* xr = x + (int64_t)b * x_s0 + (int64_t)h * x_s1;
      for (f = 0; f < F; ++f) acc[f] = 0.0;
      for (k = 0; k < K; ++k) {
        const double xv = orc_bf16_to_double(xr[k]);
        const uint16_t* wr = w + ((int64_t)h * K + k) * F;
        for (f = 0; f < F; ++f) acc[f] += xv * orc_bf16_to_double(wr[f]);
      }
      for (f = 0; f < F; ++f) {
        double v = acc[f];
        if (g) v *= 1.0 / (1.0 + exp(-orc_bf16_to_double(g[(int64_t)b * g_s0 + (int64_t)h * F + f])));
        y[((int64_t)b * H + h) * F + f] = v;
      }
    }
    free(acc);
  }
}

/* Exposed for the self-tests: the tile exponent rule and the fp32 rotation. */
int orc_ds_tile_exponent(double amax) { return ds_tile_exponent(amax); }
void orc_rope_fp32(const float* x, const float* cs_row, float* y) { rope_fp32(x, cs_row, y); }
