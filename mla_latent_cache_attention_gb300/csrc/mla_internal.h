// mla_internal.h -- parameter blocks and launchers shared by the library's translation
// units (not part of the public C ABI).
#pragma once
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace mla {

// Launch as a programmatic dependent of the previous kernel in the stream: the grid may be
// scheduled while that kernel finishes, so the kernel must execute griddepcontrol.wait before
// it touches memory that the earlier work writes (after a non-kernel operation, or a kernel
// that never triggers, this is an ordinary launch).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct AttnParams;

struct EpiParams {
  const uint16_t* ql_nope;
  int64_t ql_s0, ql_s1;
  const uint16_t* q_pe;
  int64_t qp_s0, qp_s1;
  const uint16_t* kv_c;
  int64_t kv_s0;
  const uint16_t* k_pe;
  int64_t kp_s0;
  void* mqa_q;
  uint8_t* cache;
  int64_t num_blocks, block_stride, entry_stride;
  int block_size;
  const int64_t* slot_mapping;
  const float* q_scale_inv;
  const float* cache_scale_inv;
  const int64_t* positions;
  const float* cos_sin;
  int64_t max_position;
  int H;
  int vec16;               // ql_nope rows and mqa_q 16-byte aligned (vector copies)
  uint32_t* err;
};

// Prefill epilogues: key concat + in-place q RoPE + latent insert (bf16 / fp8_ds_mla cache),
// or fp8 q / k / v quant + fp8 latent insert.
struct PrefillEpiParams {
  uint16_t* q;             // bf16 [Tp, H, dn + 64]; rotated in place (key concat) or read (fp8)
  int64_t q_s0, q_s1;
  const uint16_t* k_nope;  // bf16 [Tp, H, dn]
  int64_t kn_s0, kn_s1;
  const uint16_t* k_pe;    // bf16 [Tp, 64]
  int64_t kp_s0;
  const uint16_t* kv_c;    // bf16 [Tp, 512]
  int64_t kv_s0;
  const uint16_t* v;       // bf16 [Tp, H, dv] (fp8 only)
  int64_t v_s0, v_s1;
  uint16_t* k_out;         // bf16 [Tp, H, dn + 64] contiguous (key concat)
  uint8_t* q8;             // e4m3 [Tp, H, dn + 64], [Tp, H, dn + 64], [Tp, H, dv] contiguous (fp8)
  uint8_t* k8;
  uint8_t* v8;
  uint8_t* cache;
  int64_t num_blocks, block_stride, entry_stride;
  int block_size;
  const int64_t* slot_mapping;
  const float* q_scale_inv;  // device fp32 scalars (fp8 only)
  const float* k_scale_inv;
  const float* v_scale_inv;
  const float* cache_scale_inv;
  const int64_t* positions;
  const float* cos_sin;
  int64_t max_position;
  int H, dn, dv;
  int vec;                 // every row, stride and base 16-byte aligned: 8-element vector accesses
  uint32_t* err;
};

struct MergeParams {
  const float* part_o;     // [S][n_rows][H][512]
  const float* part_lse;   // [S][n_rows][H]
  int S, n_rows, H;
  const int32_t* seq_lens; // row r reads only the ceil(L / chunk) splits of its request r / q_len
  int q_len;
  int64_t chunk;
  uint8_t* out;            // bf16 rows
  int64_t o_s0b, o_s1b;
  float* lse;              // [n_rows, H] or null
  const float* sink;       // [H] per-head sink logit joining the denominator, or null
};

// Chunked-context gather: rows of a chunk's context entries through the block table.
struct GatherCtxParams {
  const uint8_t* cache;
  int64_t num_blocks, block_stride, entry_stride;
  int block_size;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* cu;       // [batch + 1]
  const int32_t* starts;   // [batch] or null
  int batch;
  int64_t num_tokens;
  float scale;             // plain fp8 dequantisation scale
  uint8_t* dst;
  int64_t dst_row;         // bytes
  int vec;                 // cache entries and dst rows 16-byte aligned
  uint32_t* err;
};

// merge_attn_states of a prefix and a suffix partial (bf16 [T, H, D], lse fp32 [H, T]).
struct MergeStatesParams {
  uint16_t* out;
  int64_t o_s0, o_s1;
  float* out_lse;
  const uint16_t* prefix;
  int64_t p_s0, p_s1;
  const float* prefix_lse;
  const uint16_t* suffix;
  int64_t s_s0, s_s1;
  const float* suffix_lse;
  int T, H, D;
  int vec;                 // rows 16-byte aligned, D a multiple of 8
};

// Per-head contraction y[b, h, :] = x[b, h, :K] . w[h] (w bf16 [H, K, F] contiguous), bf16
// out, optional sigmoid gate (bf16 [B, H * F] pre-activation).
struct HeadBmmParams {
  const uint16_t* x;
  int64_t x_s0, x_s1;
  const uint16_t* w;
  const uint16_t* gate;
  int64_t g_s0;
  uint16_t* y;
  int64_t y_s0, y_s1;
  int B, H, K, F;
  int vec;                 // x rows 16-byte aligned
  uint32_t* err;
};

struct GatherParams {
  const uint8_t* cache;
  int64_t num_blocks, block_stride, entry_stride;
  int block_size;
  const int64_t* slots;
  int64_t n;
  float* out;
  uint32_t* err;
};

// Set the message mla_last_error() returns on this thread.
void set_error_message(const char* msg);

cudaError_t launch_epilogue(int fmt, const EpiParams& p, int B, cudaStream_t stream);
// fmt 0 / 2: key concat for the bf16 / fp8_ds_mla cache; fmt 1: fp8 q / k / v quant.
cudaError_t launch_prefill_epilogue(int fmt, const PrefillEpiParams& p, int Tp, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_sched_reset(uint32_t* sched, cudaStream_t stream);
cudaError_t launch_gather(int fmt, const GatherParams& p, cudaStream_t stream);
// kind 0: bf16 values, 1: stored bytes
cudaError_t launch_gather_context(int fmt, int kind, const GatherCtxParams& p, cudaStream_t stream);
cudaError_t launch_merge_states(const MergeStatesParams& p, cudaStream_t stream);
// K a multiple of 64 in [64, 512], F a multiple of 128
cudaError_t launch_head_bmm(const HeadBmmParams& p, cudaStream_t stream);

// Attention launchers (one translation unit per cache format).  `grid` CTAs, each looping
// over work items; dynamic shared memory is set up on first use per device.
cudaError_t launch_attn_sparse_ds(const AttnParams& p, int grid, cudaStream_t stream);
cudaError_t launch_attn_paged_bf16(const AttnParams& p, int grid, cudaStream_t stream);
cudaError_t launch_attn_paged_fp8(const AttnParams& p, int grid, cudaStream_t stream);
cudaError_t launch_attn_paged_ds(const AttnParams& p, int grid, cudaStream_t stream);
// Paged decode with TMA page loads (ring pipeline), `nq` query columns per item.  `tkv` and
// `tq` point to CUtensorMaps: the cache as [num_blocks][block_size][entry bytes] (uint8,
// 128-byte swizzle, box 128 B x BR x 1) and the query as [rows][H][row bytes] (box 128 B x
// qbox_h x qbox_q).
struct PagedParams;
struct DsParams;
// fp8_ds_mla attention: sparse records gathered by vector loads; paged records by TMA boxes
// (`tkv` as above over the 656-byte record, `tsc` the same geometry unswizzled with 16-byte
// boxes for the scales).
cudaError_t launch_ds_sparse(const DsParams& p, int grid, cudaStream_t stream);
cudaError_t launch_ds_paged(const DsParams& p, const void* tkv, const void* tsc, int grid, cudaStream_t stream);
cudaError_t launch_ds_paged_clusters(const DsParams& p, const void* tkv, const void* tsc, int size, int clusters,
                                     cudaStream_t stream);
int ds_cluster_capacity(int size);
cudaError_t launch_paged_tma_bf16(int nq, const PagedParams& p, const void* tkv, const void* tq, int grid,
                                  cudaStream_t stream);
cudaError_t launch_paged_tma_fp8(int nq, const PagedParams& p, const void* tkv, const void* tq, int grid,
                                 cudaStream_t stream);

}  // namespace mla
