/*
 * mla.h -- C ABI of libmla: Multi-head Latent Attention over the 576-wide latent KV cache
 * on one GB300 (sm_103a).
 *
 * A cache entry is [kv_c_normed (512) | k_pe (64)], one "head" shared by all query heads
 * (MQA, num_kv_heads = 1).  Queries are absorbed to [ql_nope (512) | q_pe (64)]; the value
 * is the first 512 values of the same entry.  Three entry formats:
 *
 *   MLA_CACHE_BF16        576 bf16 values, 1152 bytes.
 *   MLA_CACHE_FP8         576 E4M3 values, 576 bytes, one per-tensor scale (k_scale).
 *   MLA_CACHE_FP8_DS_MLA  656-byte record: 512 E4M3 | 4 fp32 scales, one per 128-wide
 *                         tile of the 512 | 64 bf16 rope values ("self-scaling").
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are device memory owned by the caller; the library never
 *     allocates, frees or keeps them.  Strides are in elements of the tensor's own type
 *     unless named *_bytes; the innermost dimension is always contiguous.
 *   - Work is enqueued on `stream` (0 = legacy default stream); no call synchronises the
 *     host, except mla_read_device_errors.
 *   - Return value: MLA_OK (0); MLA_ERR_INVALID (-1) for an argument that breaks the stated
 *     contract (message in mla_last_error()); MLA_ERR_UNSUPPORTED (-2) for a shape or format
 *     outside what the kernels serve; MLA_ERR_CUDA (-3) when a launch fails.  Nothing is
 *     enqueued unless the return value is MLA_OK.  Problems of size zero return MLA_OK
 *     without launching anything.
 *   - Index checks that need device data (slot ids, block ids, positions) run inside the
 *     kernels: a bad index is skipped (masked for attention, not written for inserts) and a
 *     bit is set in the device error word, readable with mla_read_device_errors.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_CACHE_BF16 = 0,
  MLA_CACHE_FP8 = 1,
  MLA_CACHE_FP8_DS_MLA = 2
} mla_cache_format;

#define MLA_OK 0
#define MLA_ERR_INVALID (-1)
#define MLA_ERR_UNSUPPORTED (-2)
#define MLA_ERR_CUDA (-3)

/* Device error word bits (mla_read_device_errors). */
#define MLA_DEVERR_INDEX 1u       /* sparse index outside [0, num_records) that is not a masked negative */
#define MLA_DEVERR_BLOCK 2u       /* block id outside [0, num_blocks) */
#define MLA_DEVERR_SLOT 4u        /* insert slot whose block is outside [0, num_blocks) */
#define MLA_DEVERR_POSITION 8u    /* RoPE position outside [0, max_position) (clamped) */
#define MLA_DEVERR_TIMEOUT 16u    /* an in-kernel wait gave up (pipeline fault); outputs invalid */

/* Message of the last non-OK return on the calling thread ("" if none). */
MLA_API const char* mla_last_error(void);

/* Library version string. */
MLA_API const char* mla_version(void);

/* Synchronise `stream`, copy the device error word (bits above) into *flags and clear it.
 * Returns MLA_ERR_CUDA if the copy fails. */
MLA_API int mla_read_device_errors(uint32_t* flags, cudaStream_t stream);

/*
 * Profiling aid.  While both events are non-NULL, every attention-kernel launch made by
 * mla_sparse_fwd / mla_paged_decode on the calling host thread is bracketed by
 * cudaEventRecord(start) and cudaEventRecord(stop) on the call's stream (the split-K merge
 * and the epilogue are outside the bracket).  Pass NULL, NULL to stop.  The events are the
 * caller's; the library only records them.
 */
MLA_API void mla_profile_attention_events(cudaEvent_t start, cudaEvent_t stop);

/*
 * Decode epilogue: build the latent query and insert the new latent into the paged cache,
 * in one launch.
 * Follows: "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
 * fused_mla_decode_q_concat_kv_cache_insert (argument list and format dispatch), with the
 * saturating E4M3 quant of "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla"
 * (fp8_word).
 *
 *   ql_nope      device bf16 [B, H, 512], strides (ql_s0, ql_s1).
 *   q_pe         device bf16 [B, H, 64], strides (qp_s0, qp_s1).
 *   kv_c_normed  device bf16 [B, 512], row stride kv_s0.
 *   k_pe         device bf16 [B, 64] (or [B, 1, 64]), row stride kp_s0.
 *   mqa_q        device out, contiguous [B, H, 576]: bf16 for MLA_CACHE_BF16 and
 *                MLA_CACHE_FP8_DS_MLA; E4M3 bytes for MLA_CACHE_FP8, where every element is
 *                e4m3_sat(x * q_scale_inv).
 *   kv_cache     device cache: num_blocks blocks at block_stride_bytes, block_size entries
 *                each at entry_stride_bytes (>= the format's entry size).  Entry of slot s:
 *                block s / block_size, offset s % block_size.  Written in place:
 *                  BF16:   [kv_c | rope(k_pe)] as bf16;
 *                  FP8:    e4m3_sat(x * cache_scale_inv) for all 576 values;
 *                  DS_MLA: per 128-tile scale s = 2^k, k the least integer with
 *                          amax <= 448 * 2^k (s = 1 for an all-zero tile, k >= -126),
 *                          codes e4m3(x / s), scales as fp32, rope as bf16.
 *   slot_mapping device int64 [B]; a negative slot skips that token's insert (the query is
 *                still written).
 *   q_scale_inv, cache_scale_inv  device fp32 scalars; required for MLA_CACHE_FP8, must be
 *                NULL otherwise.
 *   positions    device int64 [B] and cos_sin_cache device fp32 [max_position, 64]
 *                (columns 0..31 cos, 32..63 sin): both NULL (no RoPE) or both set.  RoPE is
 *                GPT-J style on pairs (2i, 2i+1): y0 = fma(x0, c, -(x1*s)),
 *                y1 = fma(x1, c, x0*s) in fp32, applied to q_pe and k_pe before storing.
 * Errors: MLA_ERR_INVALID for NULL tensors, bad strides, mismatched scale / RoPE arguments,
 * misaligned pointers (bf16 tensors 2-byte aligned; bf16 / fp8_ds_mla cache entries
 * 4-byte aligned).
 */
MLA_API int mla_q_concat_cache_insert(const void* ql_nope, int64_t ql_s0, int64_t ql_s1,
                              const void* q_pe, int64_t qp_s0, int64_t qp_s1,
                              const void* kv_c_normed, int64_t kv_s0, const void* k_pe,
                              int64_t kp_s0, void* mqa_q, void* kv_cache, mla_cache_format fmt,
                              int64_t num_blocks, int64_t block_stride_bytes,
                              int64_t entry_stride_bytes, int32_t block_size,
                              const int64_t* slot_mapping, const float* q_scale_inv,
                              const float* cache_scale_inv, const int64_t* positions,
                              const float* cos_sin_cache, int64_t max_position, int32_t B,
                              int32_t H, cudaStream_t stream);

/*
 * Prefill epilogue for the bf16 and fp8_ds_mla caches: full per-head key, query RoPE in place
 * and latent insert, in one launch.
 * Follows: "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
 * fused_mla_key_concat_kv_cache_insert (bf16 cache) and fused_mla_key_concat_ds_mla_insert
 * (fp8_ds_mla cache).
 *
 *   q            device bf16 [Tp, H, dn + 64], strides (q_s0, q_s1); when RoPE is on its last
 *                64 values are rotated in place (bf16 of the fp32 rotation), else untouched.
 *   k_nope       device bf16 [Tp, H, dn], strides (kn_s0, kn_s1); dn a multiple of 8.
 *   k_pe         device bf16 [Tp, 64] (or [Tp, 1, 64]), row stride kp_s0.
 *   kv_c_normed  device bf16 [Tp, 512], row stride kv_s0.
 *   k_out        device out bf16 [Tp, H, dn + 64] contiguous: [k_nope[t, h] | rope(k_pe[t])]
 *                (the rotated k_pe of a token is shared by all its heads).
 *   kv_cache, fmt  MLA_CACHE_BF16 or MLA_CACHE_FP8_DS_MLA cache, geometry as in
 *                mla_q_concat_cache_insert; token t's latent [kv_c_normed | rope(k_pe)] is
 *                written at slot_mapping[t] in the same format and rounding as there (a
 *                negative slot skips it; a slot whose block is out of range is skipped and
 *                reported as MLA_DEVERR_SLOT).
 *   positions / cos_sin_cache / max_position  as in mla_q_concat_cache_insert (both NULL: no
 *                RoPE).  RoPE pairs are (2i, 2i+1) of the 64 rope values.
 * Errors: MLA_ERR_INVALID for NULL tensors, overlapping strides, misaligned (odd) bf16
 * pointers, a cache format other than the two above; MLA_ERR_UNSUPPORTED for dn not a positive
 * multiple of 8.
 */
MLA_API int mla_key_concat_cache_insert(void* q, int64_t q_s0, int64_t q_s1, const void* k_nope, int64_t kn_s0,
                                        int64_t kn_s1, const void* k_pe, int64_t kp_s0, const void* kv_c_normed,
                                        int64_t kv_s0, void* k_out, void* kv_cache, mla_cache_format fmt,
                                        int64_t num_blocks, int64_t block_stride_bytes, int64_t entry_stride_bytes,
                                        int32_t block_size, const int64_t* slot_mapping, const int64_t* positions,
                                        const float* cos_sin_cache, int64_t max_position, int32_t Tp, int32_t H,
                                        int32_t dn, cudaStream_t stream);

/*
 * Prefill epilogue for the plain fp8 cache: query, key and value quantised to E4M3, each with
 * its own scale, and the latent inserted with the cache's scale, in one launch.
 * Follows: "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
 * fused_mla_qkv_quant_kv_cache_fp8_insert (the attention key and the cache latent use separate
 * scales).  x -> e4m3_sat(x * inv) is the fp32 product rounded to nearest even on the E4M3
 * grid with saturation at +-448.
 *
 *   q, k_nope, k_pe, kv_c_normed  as in mla_key_concat_cache_insert (q is only read).
 *   v            device bf16 [Tp, H, dv], strides (v_s0, v_s1); dv a multiple of 8.
 *   q_fp8        device out E4M3 [Tp, H, dn + 64] contiguous: [q_nope | rope(q_pe)] * q_scale_inv.
 *   k_fp8        device out E4M3 [Tp, H, dn + 64] contiguous: [k_nope | rope(k_pe)] * k_scale_inv.
 *   v_fp8        device out E4M3 [Tp, H, dv] contiguous: v * v_scale_inv.
 *   kv_cache     plain fp8 cache (576-byte entries): [kv_c_normed | rope(k_pe)] * cache_scale_inv
 *                at slot_mapping[t].
 *   q_scale_inv, k_scale_inv, v_scale_inv, cache_scale_inv  device fp32 scalars (1 / scale).
 * Errors as mla_key_concat_cache_insert, plus dv.
 */
MLA_API int mla_qkv_quant_cache_fp8_insert(const void* q, int64_t q_s0, int64_t q_s1, const void* k_nope,
                                           int64_t kn_s0, int64_t kn_s1, const void* k_pe, int64_t kp_s0,
                                           const void* kv_c_normed, int64_t kv_s0, const void* v, int64_t v_s0,
                                           int64_t v_s1, void* q_fp8, void* k_fp8, void* v_fp8, void* kv_cache,
                                           int64_t num_blocks, int64_t block_stride_bytes,
                                           int64_t entry_stride_bytes, int32_t block_size,
                                           const int64_t* slot_mapping, const float* q_scale_inv,
                                           const float* k_scale_inv, const float* v_scale_inv,
                                           const float* cache_scale_inv, const int64_t* positions,
                                           const float* cos_sin_cache, int64_t max_position, int32_t Tp, int32_t H,
                                           int32_t dn, int32_t dv, cudaStream_t stream);

/*
 * Sparse MLA forward over fp8_ds_mla records with CSR key lists.
 * Follows: "vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla", flydsl_sparse_mla_fp8ds_fwd
 * (sparse_mla_fwd semantics) and flydsl_sparse_mla_fp8ds_supported (argument checks).
 *
 *   q            device bf16 [T, H, 576], strides (q_s0, q_s1) in elements, 1 <= H <= 128.
 *   kv_records   device, num_records records of 656 bytes at record_stride_bytes
 *                (a multiple of 16, >= 656; base 16-byte aligned).  Any per-128 scale is
 *                accepted (not only powers of two).
 *   kv_indptr    device int32 [T + 1], non-decreasing, kv_indptr[0] = 0.
 *   kv_indices   device int32 [n_indices], flat global record ids (n_indices < 2^31).
 *                Row t attends to kv_indices[kv_indptr[t] .. kv_indptr[t+1]); duplicates
 *                count as separate keys.  With has_invalid, entries < 0 are masked; without
 *                it every entry must be in [0, num_records) (violations are masked and
 *                reported as MLA_DEVERR_INDEX).
 *   softmax_scale  logits are softmax_scale * q.k over all 576 values.
 *   out          device bf16 [T, H, >= 512], strides (o_s0, o_s1); columns 0..511 written
 *                with softmax(logits) . V, V the 512 dequantised latent values.
 *   lse          device fp32 [T, H] contiguous, natural-log log-sum-exp of the logits over
 *                the unmasked keys; NULL to skip.
 * A row without an unmasked key gets out = 0 and lse = -inf.
 */
MLA_API int mla_sparse_fwd(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_records,
                   int64_t record_stride_bytes, int64_t num_records, const int32_t* kv_indptr,
                   const int32_t* kv_indices, int64_t n_indices, float softmax_scale,
                   int has_invalid, void* out, int64_t o_s0, int64_t o_s1, float* lse,
                   int32_t T, int32_t H, cudaStream_t stream);

/*
 * Sparse forward with the extras of the general sparse_mla_fwd: an attention sink per head, a
 * second key segment, and a split of each row's key list over several work items.
 * Follows: "vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla", flydsl_sparse_mla_fp8ds_supported
 * (the general op's argument list: attn_sink, extra_kv / extra_indptr / extra_indices,
 * kv_splits), with the semantics of flydsl_sparse_mla_fp8ds_fwd for everything else.  The page
 * names these three without defining them; this library reads them as:
 *   - attn_sink  device fp32 [H] or NULL: a logit per head (natural-log units, like
 *                softmax_scale * q.k) joining the softmax denominator with a zero value:
 *                lse = ln(sum_k e^{x_k} + e^{sink_h}), out = sum_k e^{x_k - lse} V_k; a row
 *                without keys gives out = 0 and lse = sink_h.
 *   - extra_records / extra_indptr / extra_indices  a second pool of fp8_ds_mla records (same
 *                layout rules as kv_records) with its own CSR lists over T rows: row t attends
 *                its keys of both segments under one softmax.  All NULL: no second segment.
 *   - kv_splits  in [1, 64]: each row's key list (of each segment) is cut into kv_splits
 *                contiguous parts (whole 128-key tiles) computed by separate work items and
 *                combined by their log-sum-exp; the result equals the unsplit one up to fp32
 *                rounding.
 * All other arguments as mla_sparse_fwd.  With kv_splits = 1, no sink and no second segment
 * this is mla_sparse_fwd (no workspace needed).  Otherwise `workspace` (256-byte aligned, at
 * least mla_sparse_fwd_ext_workspace_size(...) bytes, contents garbage before and after)
 * holds the fp32 partials.
 */
MLA_API size_t mla_sparse_fwd_ext_workspace_size(int32_t T, int32_t H, int32_t kv_splits, int has_extra,
                                                 int has_sink);
MLA_API int mla_sparse_fwd_ext(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_records,
                               int64_t record_stride_bytes, int64_t num_records, const int32_t* kv_indptr,
                               const int32_t* kv_indices, int64_t n_indices, const void* extra_records,
                               int64_t extra_record_stride_bytes, int64_t extra_num_records,
                               const int32_t* extra_indptr, const int32_t* extra_indices, int64_t n_extra_indices,
                               const float* attn_sink, int32_t kv_splits, float softmax_scale, int has_invalid,
                               void* out, int64_t o_s0, int64_t o_s1, float* lse, int32_t T, int32_t H,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes mla_paged_decode needs for this shape (split-K partials).  The split count
 * depends only on (B * q_len, H, max_context, the device's SM count), never on seq_lens, so
 * a graph captured once stays valid.  num_sms <= 0 means "the current device's".
 */
MLA_API size_t mla_paged_decode_workspace_size(int32_t B, int32_t q_len, int32_t H, int32_t max_context,
                                       int32_t num_sms);

/*
 * Paged MLA decode and spec-verify.
 * Follows: "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.prepared" --
 * PreparedMla.stock_core / trtllm_decode (q query tokens per request, causal among them;
 * split count bounded by max_context; bmm1_scale = softmax_scale * q_scale * k_scale and
 * bmm2_scale = k_scale for plain fp8) and pad_requests (length 0 -> zero output).
 *
 *   q            device [B * q_len, H, 576], strides (q_s0, q_s1) in elements; bf16 for the
 *                BF16 and DS_MLA caches, E4M3 bytes (raw codes, scale q_scale) for FP8.
 *                Rows are grouped by request: row b*q_len + i is request b's query i.
 *   kv_cache     device, num_blocks blocks at block_stride_bytes, block_size entries each at
 *                entry_stride_bytes (multiple of 16, >= entry size).
 *   block_table  device int32 [B, >= ceil(max seq_len / block_size)], row stride bt_stride.
 *   seq_lens     device int32 [B]: keys of request b are positions 0 .. seq_lens[b]-1 (the
 *                q_len new tokens included); query row i sees positions 0 .. L - q_len + i.
 *                0 <= seq_lens[b]; lengths beyond max_context are served but unbalanced.
 *   max_context  upper bound of seq_lens used to fix the split count (> 0).
 *   softmax_scale, q_scale, k_scale  logits = softmax_scale * q.k (BF16, DS_MLA) or
 *                softmax_scale * q_scale * k_scale * q8.k8 (FP8, raw codes), FP8 output
 *                multiplied by k_scale; q_scale / k_scale are ignored for BF16 and DS_MLA.
 *   out          device bf16 [B * q_len, H, >= 512], strides (o_s0, o_s1).
 *   lse          device fp32 [B * q_len, H] contiguous, natural log; NULL to skip.
 *   workspace    device scratch of >= mla_paged_decode_workspace_size(...) bytes, 256-byte
 *                aligned (may be NULL when that size is 0).  Contents need no initialising
 *                and are garbage afterwards.
 * A query row with no visible key gets out = 0 and lse = -inf.
 */
MLA_API int mla_paged_decode(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_cache,
                     mla_cache_format fmt, int64_t num_blocks, int64_t block_stride_bytes,
                     int64_t entry_stride_bytes, int32_t block_size, const int32_t* block_table,
                     int64_t bt_stride, const int32_t* seq_lens, int32_t B, int32_t q_len,
                     int32_t H, int32_t max_context, float softmax_scale, float q_scale,
                     float k_scale, void* out, int64_t o_s0, int64_t o_s1, float* lse,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Paged decode for callers that cannot allocate device memory.  The pages have no
 * counterpart of this entry point; it exists for callers such as code running where
 * cudaMalloc is not allowed (e.g. while a stream is being captured), plug-ins inside an engine
 * that owns all device memory and lends them none, and serving loops that forbid allocation
 * on the request path.
 *
 * Same arguments and results as mla_paged_decode, without workspace: the split-K partials go
 * to a scratch array inside the library (a file-scope __device__ buffer of 64 MiB, held on
 * every device where the library's code is loaded until the process exits).  The call
 * allocates nothing.
 *   - Shapes whose split-K scratch (mla_paged_decode_workspace_size) exceeds 64 MiB are
 *     rejected with MLA_ERR_UNSUPPORTED and a message in mla_last_error().
 *   - The first call on a device looks up the scratch's device address (once per device, with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the scratch, which keeps the previous call's contents; the decode writes
 *     every partial it reads, so nothing needs clearing.  Calls whose kernels may overlap on
 *     the GPU (e.g. on unordered streams) race on the scratch: order them.
 */
MLA_API int mla_paged_decode_noalloc(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_cache,
                                     mla_cache_format fmt, int64_t num_blocks, int64_t block_stride_bytes,
                                     int64_t entry_stride_bytes, int32_t block_size,
                                     const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                                     int32_t B, int32_t q_len, int32_t H, int32_t max_context,
                                     float softmax_scale, float q_scale, float k_scale, void* out,
                                     int64_t o_s0, int64_t o_s1, float* lse, cudaStream_t stream);

/* Output kinds of mla_gather_context. */
#define MLA_GATHER_BF16 0   /* the 576 values as bf16 */
#define MLA_GATHER_RAW 1    /* the entry bytes as stored */

/*
 * Chunked-context gather: one chunk of the requests' cached context, read through their block
 * tables into a dense workspace for the context part of a long prefill.
 * Follows: "vllm.models.kimi_k3.nvidia.mla", _compute_prefill_context / _gather_context_latent
 * (cp_gather_and_upconvert_fp8_kv_cache for fp8_ds_mla, gather_and_maybe_dequant_cache for the
 * bf16 and plain fp8 caches under a bf16 query, cp_gather_cache for plain fp8 under an fp8 query).
 *
 *   kv_cache, fmt, num_blocks, block_stride_bytes, entry_stride_bytes, block_size
 *                the paged cache, as in mla_paged_decode.
 *   block_table  device int32 [batch, >= blocks needed], row stride bt_stride: the chunk's
 *                requests' rows.
 *   cu_seq_lens  device int32 [batch + 1], non-decreasing from 0: request b fills rows
 *                cu_seq_lens[b] .. cu_seq_lens[b+1]-1 of dst.
 *   seq_starts   device int32 [batch] or NULL (all 0): row cu_seq_lens[b] + i holds context
 *                position seq_starts[b] + i of request b.
 *   num_tokens   rows of dst; rows at or past cu_seq_lens[batch] are not written.
 *   out_kind     MLA_GATHER_BF16: dst rows of 576 bf16 values -- bf16 entries as stored; plain
 *                fp8 entries e4m3 * scale; fp8_ds_mla codes e4m3 * tile scale and the bf16 rope;
 *                every product in fp32, rounded once to bf16 (round to nearest even).
 *                MLA_GATHER_RAW: dst rows of the entry bytes as stored (1152 / 576 / 656).
 *   scale        the plain fp8 cache's dequantisation scale (k_scale); unused otherwise.
 *   dst          device out, rows dst_row_stride_bytes apart.
 * A row whose block id is out of range is written as zeros and sets MLA_DEVERR_BLOCK.
 */
MLA_API int mla_gather_context(const void* kv_cache, mla_cache_format fmt, int64_t num_blocks,
                               int64_t block_stride_bytes, int64_t entry_stride_bytes, int32_t block_size,
                               const int32_t* block_table, int64_t bt_stride, const int32_t* cu_seq_lens,
                               const int32_t* seq_starts, int32_t batch, int64_t num_tokens, int32_t out_kind,
                               float scale, void* dst, int64_t dst_row_stride_bytes, cudaStream_t stream);

/*
 * Merge of two partial attentions of the same queries over disjoint key sets by their
 * log-sum-exp: the context (prefix) and new-token (suffix) parts of a chunked prefill.
 * Follows: "vllm.models.kimi_k3.nvidia.mla", _forward_prefill_fused (merge_attn_states).
 *   lse = ln(e^{lse_p} + e^{lse_s}),  output = e^{lse_p - lse} prefix + e^{lse_s - lse} suffix,
 * computed in fp32 and rounded once to bf16; both -inf -> 0 and -inf.
 *
 *   output, prefix_output, suffix_output  device bf16 [T, H, D], element strides
 *                (o_s0, o_s1) / (p_s0, p_s1) / (s_s0, s_s1), unit innermost stride.
 *   prefix_lse, suffix_lse  device fp32 [H, T] contiguous (natural log).
 *   output_lse   device fp32 [H, T] contiguous, or NULL to skip.
 */
MLA_API int mla_merge_attn_states(void* output, int64_t o_s0, int64_t o_s1, float* output_lse,
                                  const void* prefix_output, int64_t p_s0, int64_t p_s1, const float* prefix_lse,
                                  const void* suffix_output, int64_t s_s0, int64_t s_s1, const float* suffix_lse,
                                  int32_t T, int32_t H, int32_t D, cudaStream_t stream);

/*
 * Absorbed decode query: the per-head BMM1 that takes the NoPE query into the latent space
 * before the decode epilogue.
 * Follows: "vllm.models.kimi_k3.nvidia.mla", _attention (BMM1: (N, B, P) x (N, P, L) -> (B, N, L))
 * and process_weights_after_loading (W_UK_T = the key part of kv_b_proj, [N, P, L]).
 *   ql_nope[b, h, l] = sum_p q_nope[b, h, p] * w_uk_t[h, p, l]
 * on the tensor cores (bf16 operands, fp32 accumulation), rounded once to bf16.
 *
 *   q_nope   device bf16 [B, H, P], element strides (qn_s0, qn_s1), unit innermost stride
 *            (e.g. the first P values of a [B, H, P + 64] query); P in 64..512, a multiple of 64.
 *   w_uk_t   device bf16 [H, P, 512] contiguous, 16-byte aligned.
 *   ql_nope  device out bf16 [B, H, 512], element strides (ql_s0, ql_s1).
 */
MLA_API int mla_absorb_q(const void* q_nope, int64_t qn_s0, int64_t qn_s1, const void* w_uk_t, void* ql_nope,
                         int64_t ql_s0, int64_t ql_s1, int32_t B, int32_t H, int32_t P, cudaStream_t stream);

/*
 * Value up-projection of the latent attention output, with the optional output gate.
 * Follows: "vllm.models.kimi_k3.nvidia.mla", _v_up_proj ((N, B, L) x (N, L, V) -> (B, N, V))
 * and forward (_gate_sigmoid_mul of the output with the g_proj gate).
 *   y[b, h, v] = bf16(sum_l latent[b, h, l] * w_uv[h, l, v])      (fp32 accumulation)
 *   out[b, h, v] = gate ? bf16(y * bf16(sigmoid(gate[b, h * V + v]))) : y
 *
 *   latent   device bf16 [B, H, 512], element strides (l_s0, l_s1).
 *   w_uv     device bf16 [H, 512, V] contiguous, 16-byte aligned; V a multiple of 128.
 *   gate     device bf16 [B, H * V] gate pre-activations (row stride g_s0), or NULL.
 *   out      device out bf16 [B, H, V], element strides (o_s0, o_s1) (e.g. [B, H * V]).
 */
MLA_API int mla_v_up_proj(const void* latent, int64_t l_s0, int64_t l_s1, const void* w_uv, const void* gate,
                          int64_t g_s0, void* out, int64_t o_s0, int64_t o_s1, int32_t B, int32_t H, int32_t V,
                          cudaStream_t stream);

/*
 * Gather-and-dequantise (test and debugging aid): out[i, 0..575] = the exact fp32 values of
 * the entry at slots[i] (paged addressing as in mla_paged_decode; NoPE times its tile scale
 * for DS_MLA, raw E4M3 values for FP8).  Same record addressing and decode as the attention
 * kernels.  Follows "vllm.models.kimi_k3.nvidia.mla", _gather_context_latent's
 * cp_gather_and_upconvert_fp8_kv_cache (paged latent -> dense values).
 *   slots device int64 [n]; a negative slot or a bad block id gives a row of zeros.
 *   out   device fp32 [n, 576] contiguous.
 */
MLA_API int mla_gather_dequant(const void* kv_cache, mla_cache_format fmt, int64_t num_blocks,
                       int64_t block_stride_bytes, int64_t entry_stride_bytes,
                       int32_t block_size, const int64_t* slots, int64_t n, float* out,
                       cudaStream_t stream);

/*
 * Test aid: the same sparse forward as mla_sparse_fwd (same arguments, results within the
 * attention tolerance of it), computed by the second kernel design of this library: records
 * gathered by per-entry bulk copies and converted exactly to f16 in shared memory before the
 * tensor-core products.  The test-suite runs both designs on the same cases; product callers
 * use mla_sparse_fwd.
 */
MLA_API int mla_sparse_fwd_staged(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_records,
                                  int64_t record_stride_bytes, int64_t num_records, const int32_t* kv_indptr,
                                  const int32_t* kv_indices, int64_t n_indices, float softmax_scale,
                                  int has_invalid, void* out, int64_t o_s0, int64_t o_s1, float* lse,
                                  int32_t T, int32_t H, cudaStream_t stream);

/*
 * Test aid for the bounded in-kernel waits.  Arms the next mla_paged_decode call on the
 * calling host thread that runs the bf16 / plain-fp8 page kernel (block sizes 16..128 or
 * multiples of 128): that launch hands its first work item to the consumer warps but issues
 * none of its loads, and every wait in it gives up after wait_us microseconds.  The call
 * returns MLA_OK; its outputs are invalid; MLA_DEVERR_TIMEOUT is set in the device error
 * word.  No copy or tensor-core operation is in flight when the kernel exits, so the next
 * call runs normally.  wait_us <= 0 disarms.
 */
MLA_API void mla_debug_stall_next_decode(int32_t wait_us);

/*
 * Test aid: how mla_paged_decode runs an fp8_ds_mla cache on the calling host thread.  The
 * q_len * H columns of a request form G groups of 16.  size 2, 3 or 6: where size divides G,
 * the groups run as clusters of that many CTAs, which take adjacent groups of the same request
 * and split range and each issue a share of every page tile's copies with cluster multicast
 * into all of them, so each key crosses L2 -> SM once per cluster.  size 1: one CTA per group.
 * Any other value restores the library's choice (pairs where G is even).  The results are the
 * same bit for bit.
 */
MLA_API void mla_debug_ds_cluster(int32_t size);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
