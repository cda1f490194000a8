// mla_api.cu -- the C ABI declared in include/mla.h: argument checks, split-K planning,
// workspace carving and kernel launches.  Host code only; every step of the computation
// runs in the library's kernels.
#include <cuda.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "mla.h"
#include "mla_attn.cuh"
#include "mla_internal.h"
#include "mla_ds.cuh"
#include "mla_paged_tma.cuh"

namespace mla {
namespace {

__device__ uint32_t g_mla_device_errors;

thread_local char g_msg[512] = "";
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

void prof_begin(cudaStream_t s) {
  if (g_prof_start && g_prof_stop) cudaEventRecord(g_prof_start, s);
}
void prof_end(cudaStream_t s) {
  if (g_prof_start && g_prof_stop) cudaEventRecord(g_prof_stop, s);
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_msg[0] = '\0';
  return MLA_OK;
}

struct DevInfo {
  bool ready = false;
  int sms = 0;
  uint32_t* err = nullptr;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

// SM count and device error word of the current device (looked up once per device).
int dev_info(DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return fail(MLA_ERR_CUDA, "cudaGetDevice failed");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail(MLA_ERR_CUDA, "cannot query the SM count");
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mla_device_errors) != cudaSuccess)
      return fail(MLA_ERR_CUDA, "cannot resolve the device error word");
    d.err = static_cast<uint32_t*>(p);
    d.ready = true;
  }
  *out = &d;
  return MLA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int entry_bytes(mla_cache_format f) {
  return f == MLA_CACHE_BF16 ? 1152 : f == MLA_CACHE_FP8 ? 576 : 656;
}

struct SplitPlan {
  int n_splits;
  int64_t chunk;
};

// Split-K plan of the paged decode.  The split count depends on the number of (request,
// column group) units, max_context and the SM count only -- never on seq_lens -- as the
// pages' decode core fixes its split count from the deployment's longest sequence.  Aim for
// about eight work items per SM, with at least 4 key tiles (512 keys) per split; the kernels
// hand items out longest first, which evens out the tail.
SplitPlan plan_splits(int64_t units, int max_context, int sms) {
  const int64_t max_tiles = max_context > 0 ? (max_context + kTile - 1) / kTile : 1;
  int64_t splits = units > 0 ? (8LL * sms + units - 1) / units : 1;
  const int64_t cap = max_tiles / 4 > 1 ? max_tiles / 4 : 1;
  if (splits > cap) splits = cap;
  if (splits < 1) splits = 1;
  const int64_t tiles_per = (max_tiles + splits - 1) / splits;
  splits = (max_tiles + tiles_per - 1) / tiles_per;
  return SplitPlan{static_cast<int>(splits), tiles_per * kTile};
}

// Planning units: requests x groups of up to 64 query columns.
int64_t plan_units(int64_t B, int q_len, int H) {
  return B * ((static_cast<int64_t>(q_len) * H + 63) / 64);
}

// Partials [S][rows][H][512] fp32, their LSEs, and one scheduler word.
size_t workspace_bytes_for(int64_t n_rows, int H, const SplitPlan& sp) {
  if (sp.n_splits <= 1) return 0;
  const size_t po = static_cast<size_t>(sp.n_splits) * n_rows * H * kLora * sizeof(float);
  const size_t pl = static_cast<size_t>(sp.n_splits) * n_rows * H * sizeof(float);
  return ((po + 255) & ~size_t(255)) + ((pl + 255) & ~size_t(255)) + 256;
}

// Test aid: wait limit (microseconds) of the next page-kernel launch on this thread, whose
// producer then issues no loads; 0 = none armed.
thread_local int g_stall_next_us = 0;
// fp8_ds_mla paged decode: the cluster size for the head groups of a request (0: the
// library's choice; set per host thread by the test aid mla_debug_ds_cluster)
thread_local int g_ds_cluster = 0;

// Cluster size for G 16-column groups: the largest allowed size that divides G and can be
// resident, the library's default being pairs (measured best), or 1.
int ds_cluster_for(int G) {
  const int want = g_ds_cluster;
  if (want == 1 || G < 2) return 1;
  const int sizes[3] = {6, 3, 2};
  for (int sz : sizes) {
    if (want != 0 && sz != want) continue;
    if (want == 0 && sz != 2) continue;
    if (G % sz == 0 && ds_cluster_capacity(sz) > 0) return sz;
  }
  return 1;
}

int grid_for(int64_t items, int sms) {
  return static_cast<int>(items < sms ? items : sms);
}

// ---- tensor maps for the TMA page kernel (encoded through the runtime's driver entry point
// and cached by their full description; a map is only host memory passed by value)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct TmapKey {
  const void* base;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  bool swz;
  bool operator==(const TmapKey& o) const { return memcmp(this, &o, sizeof *this) == 0; }
};
struct TmapEntry {
  bool used = false;
  TmapKey key;
  CUtensorMap map;
};
TmapEntry g_tmaps[16];
int g_tmap_next = 0;
std::mutex g_tmap_mu;

// Rows per TMA box for a block size, or 0 when the page kernel does not serve it: the box
// rows must divide the 128-key tile (block_size 16..128 a power of two) or be a whole
// 128-row slice of a larger block.
int tma_rows_for(int block_size, int keys_per_tile = 128) {
  if (block_size >= keys_per_tile) return (block_size % keys_per_tile == 0) ? keys_per_tile : 0;
  if (block_size >= 16 && (keys_per_tile % block_size) == 0) return block_size;
  return 0;
}

// 3-D uint8 tensor map (128-byte swizzle, or none): dims {x bytes, y, z}, strides {y, z} in
// bytes.
int tmap_3d(const void* base, const uint64_t (&dims)[3], const uint64_t (&strides)[2], const uint32_t (&box)[3],
            CUtensorMap* out, bool swizzle = true) {
  TmapKey key{};
  key.base = base;
  key.swz = swizzle;
  for (int i = 0; i < 3; ++i) key.dims[i] = dims[i], key.box[i] = box[i];
  key.strides[0] = strides[0];
  key.strides[1] = strides[1];
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  for (auto& e : g_tmaps)
    if (e.used && e.key == key) {
      *out = e.map;
      return MLA_OK;
    }
  static EncodeTiledFn enc = nullptr;
  if (!enc) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    enc = reinterpret_cast<EncodeTiledFn>(fn);
  }
  TmapEntry& e = g_tmaps[g_tmap_next];
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides[0], strides[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), d, st, bx, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    e.used = false;
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  }
  e.used = true;
  e.key = key;
  g_tmap_next = (g_tmap_next + 1) % 16;
  *out = e.map;
  return MLA_OK;
}

// Column grouping of the page kernel: NQ query columns per item (16, 32 or 64; at most 32 for
// bf16, whose 144 KB key tiles leave less room for the query), G groups per request and the
// query box (heads x tokens) that loads one group.  Returns false when no grouping fits.
struct ColPlan {
  int nq, G, box_h, box_q;
};
bool plan_columns(int fmt, int H, int q_len, ColPlan* cp) {
  const int nqmax = fmt == MLA_CACHE_BF16 ? 32 : 64;
  const int cols = H * q_len;
  if (cols <= nqmax) {
    const int nq = cols <= 16 ? 16 : cols <= 32 ? 32 : 64;
    if (H > 256 || q_len > 256) return false;
    *cp = ColPlan{nq, 1, H, q_len};
    return true;
  }
  for (int nq = nqmax; nq >= 16; nq /= 2) {
    if (H % nq == 0) {
      *cp = ColPlan{nq, cols / nq, nq, 1};
      return true;
    }
    if (nq % H == 0) {
      const int tq = nq / H;
      *cp = ColPlan{nq, (q_len + tq - 1) / tq, H, tq};
      return true;
    }
  }
  return false;
}

}  // namespace

void set_error_message(const char* msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

}  // namespace mla

using namespace mla;

extern "C" const char* mla_last_error(void) { return g_msg; }

extern "C" const char* mla_version(void) { return "libmla 0.1 (sm_103a, tcgen05)"; }

extern "C" void mla_profile_attention_events(cudaEvent_t start, cudaEvent_t stop) {
  g_prof_start = start;
  g_prof_stop = stop;
}

extern "C" int mla_read_device_errors(uint32_t* flags, cudaStream_t stream) {
  if (!flags) return fail(MLA_ERR_INVALID, "flags is NULL");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return fail(MLA_ERR_CUDA, "stream synchronize failed");
  uint32_t v = 0;
  if (cudaMemcpy(&v, d->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "reading the device error word failed");
  const uint32_t zero = 0;
  if (cudaMemcpy(d->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "clearing the device error word failed");
  *flags = v;
  return ok();
}

// ------------------------------------------------------------------------------------------
extern "C" int mla_q_concat_cache_insert(const void* ql_nope, int64_t ql_s0, int64_t ql_s1,
                                         const void* q_pe, int64_t qp_s0, int64_t qp_s1,
                                         const void* kv_c_normed, int64_t kv_s0, const void* k_pe,
                                         int64_t kp_s0, void* mqa_q, void* kv_cache,
                                         mla_cache_format fmt, int64_t num_blocks,
                                         int64_t block_stride_bytes, int64_t entry_stride_bytes,
                                         int32_t block_size, const int64_t* slot_mapping,
                                         const float* q_scale_inv, const float* cache_scale_inv,
                                         const int64_t* positions, const float* cos_sin_cache,
                                         int64_t max_position, int32_t B, int32_t H,
                                         cudaStream_t stream) {
  if (fmt != MLA_CACHE_BF16 && fmt != MLA_CACHE_FP8 && fmt != MLA_CACHE_FP8_DS_MLA)
    return fail(MLA_ERR_INVALID, "unknown cache format %d", static_cast<int>(fmt));
  if (B < 0 || H < 1) return fail(MLA_ERR_INVALID, "bad shape B=%d H=%d", B, H);
  if (B == 0) return ok();
  if (!ql_nope || !q_pe || !kv_c_normed || !k_pe || !mqa_q || !kv_cache || !slot_mapping)
    return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (ql_s1 < 512 || ql_s0 < static_cast<int64_t>(H) * ql_s1 || qp_s1 < 64 || qp_s0 < static_cast<int64_t>(H) * qp_s1 ||
      kv_s0 < 512 || kp_s0 < 64)
    return fail(MLA_ERR_INVALID, "activation strides overlap rows");
  if (!aligned(ql_nope, 2) || !aligned(q_pe, 2) || !aligned(kv_c_normed, 2) || !aligned(k_pe, 2) || !aligned(mqa_q, 2))
    return fail(MLA_ERR_INVALID, "bf16 tensors must be 2-byte aligned");
  if (block_size < 1 || num_blocks < 1) return fail(MLA_ERR_INVALID, "bad cache geometry");
  if (entry_stride_bytes < entry_bytes(fmt) || block_stride_bytes < entry_stride_bytes * block_size)
    return fail(MLA_ERR_INVALID, "cache strides smaller than the entries");
  if (fmt != MLA_CACHE_FP8 && (entry_stride_bytes % 4 || block_stride_bytes % 4 || !aligned(kv_cache, 4)))
    return fail(MLA_ERR_INVALID, "bf16 / fp8_ds_mla cache entries must be 4-byte aligned");
  if (fmt == MLA_CACHE_FP8) {
    if (!q_scale_inv || !cache_scale_inv)
      return fail(MLA_ERR_INVALID, "the fp8 cache needs q_scale_inv and cache_scale_inv");
  } else if (q_scale_inv || cache_scale_inv) {
    return fail(MLA_ERR_INVALID, "q_scale_inv / cache_scale_inv are only for the fp8 cache");
  }
  if ((positions == nullptr) != (cos_sin_cache == nullptr))
    return fail(MLA_ERR_INVALID, "positions and cos_sin_cache must be given together");
  if (positions && max_position < 1) return fail(MLA_ERR_INVALID, "max_position must be >= 1");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  EpiParams p{};
  p.ql_nope = static_cast<const uint16_t*>(ql_nope);
  p.ql_s0 = ql_s0;
  p.ql_s1 = ql_s1;
  p.q_pe = static_cast<const uint16_t*>(q_pe);
  p.qp_s0 = qp_s0;
  p.qp_s1 = qp_s1;
  p.kv_c = static_cast<const uint16_t*>(kv_c_normed);
  p.kv_s0 = kv_s0;
  p.k_pe = static_cast<const uint16_t*>(k_pe);
  p.kp_s0 = kp_s0;
  p.mqa_q = mqa_q;
  p.cache = static_cast<uint8_t*>(kv_cache);
  p.num_blocks = num_blocks;
  p.block_stride = block_stride_bytes;
  p.entry_stride = entry_stride_bytes;
  p.block_size = block_size;
  p.slot_mapping = slot_mapping;
  p.q_scale_inv = q_scale_inv;
  p.cache_scale_inv = cache_scale_inv;
  p.positions = positions;
  p.cos_sin = cos_sin_cache;
  p.max_position = max_position;
  p.H = H;
  p.vec16 = aligned(ql_nope, 16) && aligned(mqa_q, 16) && ql_s0 % 8 == 0 && ql_s1 % 8 == 0;
  p.err = d->err;
  if (launch_epilogue(static_cast<int>(fmt), p, B, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "epilogue launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

// ------------------------------------------------------------------------------------------
// ------------------------------------------------------------------------------------------
// Prefill epilogues: shared argument checks of the key-concat and fp8-quant entry points.
static int prefill_common_checks(const void* q, int64_t q_s0, int64_t q_s1, const void* k_nope, int64_t kn_s0,
                                 int64_t kn_s1, const void* k_pe, int64_t kp_s0, const void* kv_c, int64_t kv_s0,
                                 const void* kv_cache, int fmt, int64_t num_blocks, int64_t block_stride_bytes,
                                 int64_t entry_stride_bytes, int32_t block_size, const int64_t* slot_mapping,
                                 const int64_t* positions, const float* cos_sin_cache, int64_t max_position,
                                 int32_t H, int32_t dn) {
  if (!q || !k_nope || !k_pe || !kv_c || !kv_cache || !slot_mapping)
    return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (dn < 8 || dn % 8) return fail(MLA_ERR_UNSUPPORTED, "the NoPE head dim must be a positive multiple of 8, got %d", dn);
  if (q_s1 < dn + 64 || q_s0 < static_cast<int64_t>(H) * q_s1 || kn_s1 < dn || kn_s0 < static_cast<int64_t>(H) * kn_s1 ||
      kp_s0 < 64 || kv_s0 < 512)
    return fail(MLA_ERR_INVALID, "activation strides overlap rows");
  if (!aligned(q, 2) || !aligned(k_nope, 2) || !aligned(k_pe, 2) || !aligned(kv_c, 2))
    return fail(MLA_ERR_INVALID, "bf16 tensors must be 2-byte aligned");
  if (block_size < 1 || num_blocks < 1) return fail(MLA_ERR_INVALID, "bad cache geometry");
  if (entry_stride_bytes < entry_bytes(static_cast<mla_cache_format>(fmt)) ||
      block_stride_bytes < entry_stride_bytes * block_size)
    return fail(MLA_ERR_INVALID, "cache strides smaller than the entries");
  if (fmt != MLA_CACHE_FP8 && (entry_stride_bytes % 4 || block_stride_bytes % 4 || !aligned(kv_cache, 4)))
    return fail(MLA_ERR_INVALID, "bf16 / fp8_ds_mla cache entries must be 4-byte aligned");
  if ((positions == nullptr) != (cos_sin_cache == nullptr))
    return fail(MLA_ERR_INVALID, "positions and cos_sin_cache must be given together");
  if (positions && max_position < 1) return fail(MLA_ERR_INVALID, "max_position must be >= 1");
  return MLA_OK;
}

extern "C" int mla_key_concat_cache_insert(void* q, int64_t q_s0, int64_t q_s1, const void* k_nope, int64_t kn_s0,
                                           int64_t kn_s1, const void* k_pe, int64_t kp_s0, const void* kv_c_normed,
                                           int64_t kv_s0, void* k_out, void* kv_cache, mla_cache_format fmt,
                                           int64_t num_blocks, int64_t block_stride_bytes, int64_t entry_stride_bytes,
                                           int32_t block_size, const int64_t* slot_mapping, const int64_t* positions,
                                           const float* cos_sin_cache, int64_t max_position, int32_t Tp, int32_t H,
                                           int32_t dn, cudaStream_t stream) {
  if (fmt != MLA_CACHE_BF16 && fmt != MLA_CACHE_FP8_DS_MLA)
    return fail(MLA_ERR_INVALID, "the key-concat epilogue writes a bf16 or fp8_ds_mla cache (format %d)",
                static_cast<int>(fmt));
  if (Tp < 0 || H < 1) return fail(MLA_ERR_INVALID, "bad shape Tp=%d H=%d", Tp, H);
  if (Tp == 0) return ok();
  if (int rc = prefill_common_checks(q, q_s0, q_s1, k_nope, kn_s0, kn_s1, k_pe, kp_s0, kv_c_normed, kv_s0, kv_cache,
                                     fmt, num_blocks, block_stride_bytes, entry_stride_bytes, block_size, slot_mapping,
                                     positions, cos_sin_cache, max_position, H, dn))
    return rc;
  if (!k_out) return fail(MLA_ERR_INVALID, "k_out is NULL");
  if (!aligned(k_out, 2)) return fail(MLA_ERR_INVALID, "k_out must be 2-byte aligned");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  PrefillEpiParams p{};
  p.q = static_cast<uint16_t*>(q);
  p.q_s0 = q_s0;
  p.q_s1 = q_s1;
  p.k_nope = static_cast<const uint16_t*>(k_nope);
  p.kn_s0 = kn_s0;
  p.kn_s1 = kn_s1;
  p.k_pe = static_cast<const uint16_t*>(k_pe);
  p.kp_s0 = kp_s0;
  p.kv_c = static_cast<const uint16_t*>(kv_c_normed);
  p.kv_s0 = kv_s0;
  p.k_out = static_cast<uint16_t*>(k_out);
  p.cache = static_cast<uint8_t*>(kv_cache);
  p.num_blocks = num_blocks;
  p.block_stride = block_stride_bytes;
  p.entry_stride = entry_stride_bytes;
  p.block_size = block_size;
  p.slot_mapping = slot_mapping;
  p.positions = positions;
  p.cos_sin = cos_sin_cache;
  p.max_position = max_position;
  p.H = H;
  p.dn = dn;
  p.vec = aligned(k_nope, 16) && aligned(k_out, 16) && kn_s0 % 8 == 0 && kn_s1 % 8 == 0;
  p.err = d->err;
  if (launch_prefill_epilogue(static_cast<int>(fmt), p, Tp, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "prefill epilogue launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

extern "C" int mla_qkv_quant_cache_fp8_insert(const void* q, int64_t q_s0, int64_t q_s1, const void* k_nope,
                                              int64_t kn_s0, int64_t kn_s1, const void* k_pe, int64_t kp_s0,
                                              const void* kv_c_normed, int64_t kv_s0, const void* v, int64_t v_s0,
                                              int64_t v_s1, void* q_fp8, void* k_fp8, void* v_fp8, void* kv_cache,
                                              int64_t num_blocks, int64_t block_stride_bytes,
                                              int64_t entry_stride_bytes, int32_t block_size,
                                              const int64_t* slot_mapping, const float* q_scale_inv,
                                              const float* k_scale_inv, const float* v_scale_inv,
                                              const float* cache_scale_inv, const int64_t* positions,
                                              const float* cos_sin_cache, int64_t max_position, int32_t Tp, int32_t H,
                                              int32_t dn, int32_t dv, cudaStream_t stream) {
  if (Tp < 0 || H < 1) return fail(MLA_ERR_INVALID, "bad shape Tp=%d H=%d", Tp, H);
  if (Tp == 0) return ok();
  if (int rc = prefill_common_checks(q, q_s0, q_s1, k_nope, kn_s0, kn_s1, k_pe, kp_s0, kv_c_normed, kv_s0, kv_cache,
                                     MLA_CACHE_FP8, num_blocks, block_stride_bytes, entry_stride_bytes, block_size,
                                     slot_mapping, positions, cos_sin_cache, max_position, H, dn))
    return rc;
  if (!v || !q_fp8 || !k_fp8 || !v_fp8 || !q_scale_inv || !k_scale_inv || !v_scale_inv || !cache_scale_inv)
    return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (dv < 8 || dv % 8) return fail(MLA_ERR_UNSUPPORTED, "the value head dim must be a positive multiple of 8, got %d", dv);
  if (v_s1 < dv || v_s0 < static_cast<int64_t>(H) * v_s1) return fail(MLA_ERR_INVALID, "v strides overlap rows");
  if (!aligned(v, 2)) return fail(MLA_ERR_INVALID, "v must be 2-byte aligned");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  PrefillEpiParams p{};
  p.q = const_cast<uint16_t*>(static_cast<const uint16_t*>(q));   // read only for the fp8 epilogue
  p.q_s0 = q_s0;
  p.q_s1 = q_s1;
  p.k_nope = static_cast<const uint16_t*>(k_nope);
  p.kn_s0 = kn_s0;
  p.kn_s1 = kn_s1;
  p.k_pe = static_cast<const uint16_t*>(k_pe);
  p.kp_s0 = kp_s0;
  p.kv_c = static_cast<const uint16_t*>(kv_c_normed);
  p.kv_s0 = kv_s0;
  p.v = static_cast<const uint16_t*>(v);
  p.v_s0 = v_s0;
  p.v_s1 = v_s1;
  p.q8 = static_cast<uint8_t*>(q_fp8);
  p.k8 = static_cast<uint8_t*>(k_fp8);
  p.v8 = static_cast<uint8_t*>(v_fp8);
  p.cache = static_cast<uint8_t*>(kv_cache);
  p.num_blocks = num_blocks;
  p.block_stride = block_stride_bytes;
  p.entry_stride = entry_stride_bytes;
  p.block_size = block_size;
  p.slot_mapping = slot_mapping;
  p.q_scale_inv = q_scale_inv;
  p.k_scale_inv = k_scale_inv;
  p.v_scale_inv = v_scale_inv;
  p.cache_scale_inv = cache_scale_inv;
  p.positions = positions;
  p.cos_sin = cos_sin_cache;
  p.max_position = max_position;
  p.H = H;
  p.dn = dn;
  p.dv = dv;
  p.vec = aligned(q, 16) && aligned(k_nope, 16) && aligned(v, 16) && aligned(q_fp8, 8) && aligned(k_fp8, 8) &&
          aligned(v_fp8, 8) && q_s0 % 8 == 0 && q_s1 % 8 == 0 && kn_s0 % 8 == 0 && kn_s1 % 8 == 0 && v_s0 % 8 == 0 &&
          v_s1 % 8 == 0;
  p.err = d->err;
  if (launch_prefill_epilogue(1, p, Tp, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "prefill epilogue launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

// The sparse forward: the gather-warp fp8_ds_mla kernel (codes straight into the tensor
// cores), or for the test aid mla_sparse_fwd_staged the staged-converter kernel (codes
// converted to f16 in shared memory).
static int sparse_fwd_impl(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_records,
                           int64_t record_stride_bytes, int64_t num_records, const int32_t* kv_indptr,
                           const int32_t* kv_indices, int64_t n_indices, float softmax_scale, int has_invalid,
                           void* out, int64_t o_s0, int64_t o_s1, float* lse, int32_t T, int32_t H,
                           cudaStream_t stream, bool staged) {
  if (T < 0) return fail(MLA_ERR_INVALID, "T must be >= 0");
  if (H < 1 || H > 128) return fail(MLA_ERR_UNSUPPORTED, "H must be in [1, 128], got %d", H);
  if (T == 0) return ok();
  if (!q || !kv_records || !kv_indptr || !out) return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (n_indices < 0 || n_indices >= (int64_t(1) << 31))
    return fail(MLA_ERR_UNSUPPORTED, "n_indices must be in [0, 2^31)");
  if (n_indices > 0 && !kv_indices) return fail(MLA_ERR_INVALID, "kv_indices is NULL");
  if (num_records < 1) return fail(MLA_ERR_INVALID, "num_records must be >= 1");
  if (record_stride_bytes < 656 || record_stride_bytes % 16 || !aligned(kv_records, 16))
    return fail(MLA_ERR_INVALID, "records need a 16-byte aligned base and a pitch that is a multiple of 16 (>= 656)");
  if (!aligned(q, 16) || q_s1 < 576 || q_s1 % 8 || q_s0 % 8 || q_s0 < static_cast<int64_t>(H) * q_s1)
    return fail(MLA_ERR_INVALID, "q must be 16-byte aligned with strides that are multiples of 8 elements");
  if (!aligned(out, 2) || o_s1 < 512 || o_s0 < static_cast<int64_t>(H) * o_s1)
    return fail(MLA_ERR_INVALID, "bad out strides");
  if (lse && !aligned(lse, 4)) return fail(MLA_ERR_INVALID, "lse must be 4-byte aligned");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  DsParams p{};
  p.q = static_cast<const uint8_t*>(q);
  p.q_s0b = q_s0 * 2;
  p.q_s1b = q_s1 * 2;
  p.H = H;
  p.q_len = 1;
  p.B = T;
  p.G = (H + 15) / 16;
  p.cols = H;
  p.records = static_cast<const uint8_t*>(kv_records);
  p.rec_stride = record_stride_bytes;
  p.num_records = num_records;
  p.indptr = kv_indptr;
  p.indices = kv_indices;
  p.has_invalid = has_invalid ? 1 : 0;
  p.chunk = 0;
  p.n_splits = 1;
  p.n_rows = T;
  const int64_t items = static_cast<int64_t>(T) * p.G;
  if (items >= (int64_t(1) << 31)) return fail(MLA_ERR_UNSUPPORTED, "too many work items");
  p.n_items = static_cast<int>(items);
  p.sig2 = softmax_scale * 1.4426950408889634f;
  p.out = static_cast<uint8_t*>(out);
  p.o_s0b = o_s0 * 2;
  p.o_s1b = o_s1 * 2;
  p.lse = lse;
  p.sched = nullptr;
  p.err = d->err;
  prof_begin(stream);
  cudaError_t e;
  if (!staged) {
    e = launch_ds_sparse(p, grid_for(items, d->sms), stream);
  } else {
    AttnParams a{};
    a.q = p.q;
    a.q_s0b = p.q_s0b;
    a.q_s1b = p.q_s1b;
    a.H = H;
    a.n_hgroups = (H + kRows - 1) / kRows;
    a.records = p.records;
    a.rec_stride = p.rec_stride;
    a.num_records = p.num_records;
    a.indptr = p.indptr;
    a.indices = p.indices;
    a.has_invalid = p.has_invalid;
    a.q_len = 1;
    a.n_splits = 1;
    a.chunk = 0;
    a.n_rows = T;
    a.n_items = T * a.n_hgroups;
    a.sig2 = p.sig2;
    a.out_scale = 1.f;
    a.out = p.out;
    a.o_s0b = p.o_s0b;
    a.o_s1b = p.o_s1b;
    a.lse = lse;
    a.err = d->err;
    e = launch_attn_sparse_ds(a, grid_for(a.n_items, d->sms), stream);
  }
  prof_end(stream);
  if (e != cudaSuccess)
    return fail(MLA_ERR_CUDA, "sparse attention launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

extern "C" int mla_sparse_fwd(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_records,
                              int64_t record_stride_bytes, int64_t num_records,
                              const int32_t* kv_indptr, const int32_t* kv_indices, int64_t n_indices,
                              float softmax_scale, int has_invalid, void* out, int64_t o_s0,
                              int64_t o_s1, float* lse, int32_t T, int32_t H, cudaStream_t stream) {
  return sparse_fwd_impl(q, q_s0, q_s1, kv_records, record_stride_bytes, num_records, kv_indptr, kv_indices,
                         n_indices, softmax_scale, has_invalid, out, o_s0, o_s1, lse, T, H, stream, false);
}

extern "C" int mla_sparse_fwd_staged(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_records,
                                     int64_t record_stride_bytes, int64_t num_records,
                                     const int32_t* kv_indptr, const int32_t* kv_indices, int64_t n_indices,
                                     float softmax_scale, int has_invalid, void* out, int64_t o_s0,
                                     int64_t o_s1, float* lse, int32_t T, int32_t H, cudaStream_t stream) {
  return sparse_fwd_impl(q, q_s0, q_s1, kv_records, record_stride_bytes, num_records, kv_indptr, kv_indices,
                         n_indices, softmax_scale, has_invalid, out, o_s0, o_s1, lse, T, H, stream, true);
}

// ------------------------------------------------------------------------------------------
// Sparse forward with the general op's extras.  Every launch of the gather-warp kernel writes
// fp32 partials (one per split and segment) into the workspace; the LSE merge kernel combines
// them (and the sink) into out / lse.
static size_t sparse_ext_partials(int32_t kv_splits, bool has_extra) {
  return static_cast<size_t>(kv_splits) * (has_extra ? 2 : 1);
}

extern "C" size_t mla_sparse_fwd_ext_workspace_size(int32_t T, int32_t H, int32_t kv_splits, int has_extra,
                                                    int has_sink) {
  if (T <= 0 || H <= 0 || kv_splits < 1) return 0;
  const size_t S = sparse_ext_partials(kv_splits, has_extra != 0);
  if (S == 1 && !has_sink) return 0;
  return workspace_bytes_for(T, H, SplitPlan{static_cast<int>(S < 2 ? 2 : S), 0});
}

extern "C" int mla_sparse_fwd_ext(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_records,
                                  int64_t record_stride_bytes, int64_t num_records, const int32_t* kv_indptr,
                                  const int32_t* kv_indices, int64_t n_indices, const void* extra_records,
                                  int64_t extra_record_stride_bytes, int64_t extra_num_records,
                                  const int32_t* extra_indptr, const int32_t* extra_indices, int64_t n_extra_indices,
                                  const float* attn_sink, int32_t kv_splits, float softmax_scale, int has_invalid,
                                  void* out, int64_t o_s0, int64_t o_s1, float* lse, int32_t T, int32_t H,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const bool has_extra = extra_records != nullptr;
  if (has_extra != (extra_indptr != nullptr))
    return fail(MLA_ERR_INVALID, "extra_records and extra_indptr must be given together");
  if (kv_splits < 1 || kv_splits > 64) return fail(MLA_ERR_UNSUPPORTED, "kv_splits must be in [1, 64], got %d", kv_splits);
  const size_t S = sparse_ext_partials(kv_splits, has_extra);
  if (S == 1 && !attn_sink)       // nothing beyond the plain forward
    return sparse_fwd_impl(q, q_s0, q_s1, kv_records, record_stride_bytes, num_records, kv_indptr, kv_indices,
                           n_indices, softmax_scale, has_invalid, out, o_s0, o_s1, lse, T, H, stream, false);
  if (T < 0) return fail(MLA_ERR_INVALID, "T must be >= 0");
  if (H < 1 || H > 128) return fail(MLA_ERR_UNSUPPORTED, "H must be in [1, 128], got %d", H);
  if (T == 0) return ok();
  if (!q || !kv_records || !kv_indptr || !out) return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (n_indices < 0 || n_indices >= (int64_t(1) << 31) || n_extra_indices < 0 || n_extra_indices >= (int64_t(1) << 31))
    return fail(MLA_ERR_UNSUPPORTED, "index counts must be in [0, 2^31)");
  if ((n_indices > 0 && !kv_indices) || (has_extra && n_extra_indices > 0 && !extra_indices))
    return fail(MLA_ERR_INVALID, "an index array is NULL");
  if (num_records < 1 || (has_extra && extra_num_records < 1)) return fail(MLA_ERR_INVALID, "num_records must be >= 1");
  if (record_stride_bytes < 656 || record_stride_bytes % 16 || !aligned(kv_records, 16) ||
      (has_extra && (extra_record_stride_bytes < 656 || extra_record_stride_bytes % 16 || !aligned(extra_records, 16))))
    return fail(MLA_ERR_INVALID, "records need a 16-byte aligned base and a pitch that is a multiple of 16 (>= 656)");
  if (!aligned(q, 16) || q_s1 < 576 || q_s1 % 8 || q_s0 % 8 || q_s0 < static_cast<int64_t>(H) * q_s1)
    return fail(MLA_ERR_INVALID, "q must be 16-byte aligned with strides that are multiples of 8 elements");
  if (!aligned(out, 2) || o_s1 < 512 || o_s0 < static_cast<int64_t>(H) * o_s1)
    return fail(MLA_ERR_INVALID, "bad out strides");
  if (lse && !aligned(lse, 4)) return fail(MLA_ERR_INVALID, "lse must be 4-byte aligned");
  if (attn_sink && !aligned(attn_sink, 4)) return fail(MLA_ERR_INVALID, "attn_sink must be 4-byte aligned");
  const size_t need = mla_sparse_fwd_ext_workspace_size(T, H, kv_splits, has_extra ? 1 : 0, attn_sink ? 1 : 0);
  if (!workspace || workspace_bytes < need)
    return fail(MLA_ERR_INVALID, "workspace too small: need %zu bytes, got %zu", need, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(MLA_ERR_INVALID, "workspace must be 256-byte aligned");
  const int G = (H + 15) / 16;
  const int64_t items = static_cast<int64_t>(kv_splits) * T * G;
  if (items >= (int64_t(1) << 31)) return fail(MLA_ERR_UNSUPPORTED, "too many work items");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  const size_t po = S * static_cast<size_t>(T) * H * kLora * sizeof(float);
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ((po + 255) & ~size_t(255)));
  prof_begin(stream);
  for (int seg = 0; seg < (has_extra ? 2 : 1); ++seg) {
    DsParams p{};
    p.q = static_cast<const uint8_t*>(q);
    p.q_s0b = q_s0 * 2;
    p.q_s1b = q_s1 * 2;
    p.H = H;
    p.q_len = 1;
    p.B = T;
    p.G = G;
    p.cols = H;
    p.records = static_cast<const uint8_t*>(seg ? extra_records : kv_records);
    p.rec_stride = seg ? extra_record_stride_bytes : record_stride_bytes;
    p.num_records = seg ? extra_num_records : num_records;
    p.indptr = seg ? extra_indptr : kv_indptr;
    p.indices = seg ? extra_indices : kv_indices;
    p.has_invalid = has_invalid ? 1 : 0;
    p.n_splits = kv_splits;
    p.n_rows = T;
    p.n_items = static_cast<int>(items);
    p.sig2 = softmax_scale * 1.4426950408889634f;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.err = d->err;
    p.partial = 1;
    p.split_base = seg * kv_splits;
    if (launch_ds_sparse(p, grid_for(items, d->sms), stream) != cudaSuccess) {
      prof_end(stream);
      return fail(MLA_ERR_CUDA, "sparse attention launch failed: %s", cudaGetErrorString(cudaGetLastError()));
    }
  }
  prof_end(stream);
  MergeParams m{};
  m.part_o = part_o;
  m.part_lse = part_lse;
  m.S = static_cast<int>(S);
  m.n_rows = T;
  m.H = H;
  m.seq_lens = nullptr;
  m.q_len = 1;
  m.chunk = 1;
  m.out = static_cast<uint8_t*>(out);
  m.o_s0b = o_s0 * 2;
  m.o_s1b = o_s1 * 2;
  m.lse = lse;
  m.sink = attn_sink;
  if (launch_merge(m, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "merge launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

extern "C" void mla_debug_stall_next_decode(int32_t wait_us) { g_stall_next_us = wait_us > 0 ? wait_us : 0; }

extern "C" void mla_debug_ds_cluster(int32_t size) {
  g_ds_cluster = (size == 1 || size == 2 || size == 3 || size == 6) ? size : 0;
}

// ------------------------------------------------------------------------------------------
extern "C" size_t mla_paged_decode_workspace_size(int32_t B, int32_t q_len, int32_t H,
                                                  int32_t max_context, int32_t num_sms) {
  if (B <= 0 || q_len <= 0 || H <= 0 || max_context <= 0) return 0;
  int sms = num_sms;
  if (sms <= 0) {
    DevInfo* d = nullptr;
    if (dev_info(&d) != MLA_OK) return 0;
    sms = d->sms;
  }
  const int64_t n_rows = static_cast<int64_t>(B) * q_len;
  const SplitPlan sp = plan_splits(plan_units(B, q_len, H), max_context, sms);
  return workspace_bytes_for(n_rows, H, sp);
}

extern "C" int mla_paged_decode(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_cache,
                                mla_cache_format fmt, int64_t num_blocks, int64_t block_stride_bytes,
                                int64_t entry_stride_bytes, int32_t block_size,
                                const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                                int32_t B, int32_t q_len, int32_t H, int32_t max_context,
                                float softmax_scale, float q_scale, float k_scale, void* out,
                                int64_t o_s0, int64_t o_s1, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  if (fmt != MLA_CACHE_BF16 && fmt != MLA_CACHE_FP8 && fmt != MLA_CACHE_FP8_DS_MLA)
    return fail(MLA_ERR_INVALID, "unknown cache format %d", static_cast<int>(fmt));
  if (B < 0 || q_len < 1 || H < 1) return fail(MLA_ERR_INVALID, "bad shape B=%d q_len=%d H=%d", B, q_len, H);
  if (H > 128) return fail(MLA_ERR_UNSUPPORTED, "H must be <= 128, got %d", H);
  if (max_context < 1) return fail(MLA_ERR_INVALID, "max_context must be >= 1");
  if (B == 0) return ok();
  if (!q || !kv_cache || !block_table || !seq_lens || !out) return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (block_size < 1 || num_blocks < 1 || bt_stride < 1) return fail(MLA_ERR_INVALID, "bad cache geometry");
  if (entry_stride_bytes < entry_bytes(fmt) || entry_stride_bytes % 16 || block_stride_bytes % 16 ||
      block_stride_bytes < entry_stride_bytes * block_size || !aligned(kv_cache, 16))
    return fail(MLA_ERR_INVALID, "cache entries need 16-byte alignment and non-overlapping strides");
  const int qalign = fmt == MLA_CACHE_FP8 ? 8 : 16;
  if (!aligned(q, qalign) || q_s1 < 576 || q_s1 % 8 || q_s0 % 8 || q_s0 < static_cast<int64_t>(H) * q_s1)
    return fail(MLA_ERR_INVALID, "q must be %d-byte aligned with strides that are multiples of 8 elements", qalign);
  if (!aligned(out, 2) || o_s1 < 512 || o_s0 < static_cast<int64_t>(H) * o_s1)
    return fail(MLA_ERR_INVALID, "bad out strides");
  if (lse && !aligned(lse, 4)) return fail(MLA_ERR_INVALID, "lse must be 4-byte aligned");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  const int64_t n_rows = static_cast<int64_t>(B) * q_len;
  const int n_hgroups = (H + kRows - 1) / kRows;
  const SplitPlan sp = plan_splits(plan_units(B, q_len, H), max_context, d->sms);
  const size_t need = workspace_bytes_for(n_rows, H, sp);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return fail(MLA_ERR_INVALID, "workspace too small: need %zu bytes, got %zu", need, workspace_bytes);
    if (!aligned(workspace, 256)) return fail(MLA_ERR_INVALID, "workspace must be 256-byte aligned");
  }
  float* part_o = nullptr;
  float* part_lse = nullptr;
  uint32_t* sched = nullptr;
  if (sp.n_splits > 1) {
    const size_t po = static_cast<size_t>(sp.n_splits) * n_rows * H * kLora * sizeof(float);
    const size_t pl = static_cast<size_t>(sp.n_splits) * n_rows * H * sizeof(float);
    part_o = static_cast<float*>(workspace);
    part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ((po + 255) & ~size_t(255)));
    sched = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + ((po + 255) & ~size_t(255)) +
                                        ((pl + 255) & ~size_t(255)));
  }
  const float sigma = fmt == MLA_CACHE_FP8 ? softmax_scale * q_scale * k_scale : softmax_scale;
  const float out_scale = fmt == MLA_CACHE_FP8 ? k_scale : 1.f;
  const int qe = fmt == MLA_CACHE_FP8 ? 1 : 2;

  // The TMA page kernels serve caches whose blocks tile the 128-key tile, with a query whose
  // rows and heads are 16-byte aligned.
  const int tma_rows = tma_rows_for(block_size);
  if (fmt == MLA_CACHE_FP8_DS_MLA && tma_rows > 0 && aligned(q, 16) && (q_s0 * 2) % 16 == 0 && (q_s1 * 2) % 16 == 0 &&
      num_blocks < (int64_t(1) << 31) && max_context < (1 << 30)) {
    const int G = (q_len * H + 15) / 16;
    // head groups of a request run as a cluster of CTAs that share each page tile
    const int csize = ds_cluster_for(G);
    const int64_t items = static_cast<int64_t>(sp.n_splits) * B * (G / csize);
    if (items >= (int64_t(1) << 31)) return fail(MLA_ERR_UNSUPPORTED, "too many work items");
    CUtensorMap tkv, tsc;
    const uint64_t kd[3] = {656, static_cast<uint64_t>(block_size), static_cast<uint64_t>(num_blocks)};
    const uint64_t ks[2] = {static_cast<uint64_t>(entry_stride_bytes), static_cast<uint64_t>(block_stride_bytes)};
    const uint32_t kb[3] = {128, static_cast<uint32_t>(tma_rows), 1};
    const uint32_t sb[3] = {16, static_cast<uint32_t>(tma_rows), 1};
    if (int rc = tmap_3d(kv_cache, kd, ks, kb, &tkv)) return rc;
    if (int rc = tmap_3d(kv_cache, kd, ks, sb, &tsc, false)) return rc;
    DsParams p{};
    p.q = static_cast<const uint8_t*>(q);
    p.q_s0b = q_s0 * 2;
    p.q_s1b = q_s1 * 2;
    p.H = H;
    p.q_len = q_len;
    p.B = B;
    p.G = G;
    p.cols = H * q_len;
    p.block_table = block_table;
    p.bt_stride = bt_stride;
    p.seq_lens = seq_lens;
    p.num_blocks = static_cast<int>(num_blocks);
    p.block_size = block_size;
    p.BR = tma_rows;
    p.chunk = static_cast<int>(sp.chunk);
    p.n_splits = sp.n_splits;
    p.n_items = static_cast<int>(items);
    p.n_rows = static_cast<int>(n_rows);
    p.sig2 = softmax_scale * 1.4426950408889634f;
    p.out = static_cast<uint8_t*>(out);
    p.o_s0b = o_s0 * 2;
    p.o_s1b = o_s1 * 2;
    p.lse = lse;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.sched = sched;
    p.err = d->err;
    p.partial = sp.n_splits > 1 ? 1 : 0;
    if (sched && launch_sched_reset(sched, stream) != cudaSuccess)
      return fail(MLA_ERR_CUDA, "scheduler reset failed: %s", cudaGetErrorString(cudaGetLastError()));
    prof_begin(stream);
    const cudaError_t e =
        csize > 1 ? launch_ds_paged_clusters(p, &tkv, &tsc, csize, grid_for(items, ds_cluster_capacity(csize)), stream)
                  : launch_ds_paged(p, &tkv, &tsc, grid_for(items, d->sms), stream);
    prof_end(stream);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "decode attention launch failed: %s", cudaGetErrorString(e));
    if (sp.n_splits > 1) {
      MergeParams m{};
      m.part_o = part_o;
      m.part_lse = part_lse;
      m.S = sp.n_splits;
      m.n_rows = static_cast<int>(n_rows);
      m.H = H;
      m.seq_lens = seq_lens;
      m.q_len = q_len;
      m.chunk = sp.chunk;
      m.out = static_cast<uint8_t*>(out);
      m.o_s0b = o_s0 * 2;
      m.o_s1b = o_s1 * 2;
      m.lse = lse;
      if (launch_merge(m, stream) != cudaSuccess)
        return fail(MLA_ERR_CUDA, "merge launch failed: %s", cudaGetErrorString(cudaGetLastError()));
    }
    return ok();
  }
  const bool tma_fmt = fmt != MLA_CACHE_FP8_DS_MLA;
  // keys per tile of the page kernel (a template choice; 128 for both formats, measured
  // faster than 64-key tiles for bf16 despite the deeper ring those allow)
  const int tma_rows_p = tma_rows_for(block_size, 128);
  ColPlan cp{};
  const bool use_tma = tma_fmt && tma_rows_p > 0 && plan_columns(static_cast<int>(fmt), H, q_len, &cp) && aligned(q, 16) &&
                       (q_s0 * qe) % 16 == 0 && (q_s1 * qe) % 16 == 0 && num_blocks < (int64_t(1) << 31) &&
                       max_context < (1 << 30);
  cudaError_t e;
  if (use_tma) {
    const int64_t items = static_cast<int64_t>(sp.n_splits) * B * cp.G;
    if (items >= (int64_t(1) << 31)) return fail(MLA_ERR_UNSUPPORTED, "too many work items");
    CUtensorMap tkv, tq;
    const uint64_t kd[3] = {static_cast<uint64_t>(entry_bytes(fmt)), static_cast<uint64_t>(block_size),
                            static_cast<uint64_t>(num_blocks)};
    const uint64_t ks[2] = {static_cast<uint64_t>(entry_stride_bytes), static_cast<uint64_t>(block_stride_bytes)};
    const uint32_t kb[3] = {128, static_cast<uint32_t>(tma_rows_p), 1};
    if (int rc = tmap_3d(kv_cache, kd, ks, kb, &tkv)) return rc;
    const uint64_t qd[3] = {static_cast<uint64_t>(576 * qe), static_cast<uint64_t>(H), static_cast<uint64_t>(n_rows)};
    const uint64_t qs[2] = {static_cast<uint64_t>(q_s1 * qe), static_cast<uint64_t>(q_s0 * qe)};
    const uint32_t qb[3] = {128, static_cast<uint32_t>(cp.box_h), static_cast<uint32_t>(cp.box_q)};
    if (int rc = tmap_3d(q, qd, qs, qb, &tq)) return rc;
    PagedParams p{};
    p.kv = static_cast<const uint8_t*>(kv_cache);
    p.kv_blk_stride = block_stride_bytes;
    p.kv_ent_stride = entry_stride_bytes;
    p.H = H;
    p.q_len = q_len;
    p.B = B;
    p.G = cp.G;
    p.cols = H * q_len;
    p.qbox_h = cp.box_h;
    p.qbox_q = cp.box_q;
    p.block_table = block_table;
    p.bt_stride = bt_stride;
    p.seq_lens = seq_lens;
    p.num_blocks = static_cast<int>(num_blocks);
    p.block_size = block_size;
    p.BR = tma_rows_p;
    p.chunk = static_cast<int>(sp.chunk);
    p.n_splits = sp.n_splits;
    p.n_items = static_cast<int>(items);
    p.n_rows = static_cast<int>(n_rows);
    p.sig2 = sigma * 1.4426950408889634f;
    p.out_scale = out_scale;
    p.out = static_cast<uint8_t*>(out);
    p.o_s0b = o_s0 * 2;
    p.o_s1b = o_s1 * 2;
    p.lse = lse;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.sched = sched;
    p.err = d->err;
    p.wait_us = g_stall_next_us;
    p.stall = g_stall_next_us > 0 ? 1 : 0;
    g_stall_next_us = 0;
    if (sched && launch_sched_reset(sched, stream) != cudaSuccess)
      return fail(MLA_ERR_CUDA, "scheduler reset failed: %s", cudaGetErrorString(cudaGetLastError()));
    const int grid = grid_for(items, d->sms);
    prof_begin(stream);
    e = fmt == MLA_CACHE_BF16 ? launch_paged_tma_bf16(cp.nq, p, &tkv, &tq, grid, stream)
                              : launch_paged_tma_fp8(cp.nq, p, &tkv, &tq, grid, stream);
    prof_end(stream);
  } else {
    const int64_t items = n_rows * n_hgroups * sp.n_splits;
    if (items >= (int64_t(1) << 31)) return fail(MLA_ERR_UNSUPPORTED, "too many work items");
    AttnParams p{};
    p.q = static_cast<const uint8_t*>(q);
    p.q_s0b = q_s0 * qe;
    p.q_s1b = q_s1 * qe;
    p.H = H;
    p.n_hgroups = n_hgroups;
    p.cache = static_cast<const uint8_t*>(kv_cache);
    p.num_blocks = num_blocks;
    p.block_stride = block_stride_bytes;
    p.entry_stride = entry_stride_bytes;
    p.block_size = block_size;
    p.block_table = block_table;
    p.bt_stride = bt_stride;
    p.seq_lens = seq_lens;
    p.q_len = q_len;
    p.chunk = sp.chunk;
    p.n_splits = sp.n_splits;
    p.n_rows = static_cast<int>(n_rows);
    p.n_items = static_cast<int>(items);
    p.sig2 = sigma * 1.4426950408889634f;
    p.out_scale = out_scale;
    p.out = static_cast<uint8_t*>(out);
    p.o_s0b = o_s0 * 2;
    p.o_s1b = o_s1 * 2;
    p.lse = lse;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.err = d->err;
    const int grid = grid_for(items, d->sms);
    prof_begin(stream);
    if (fmt == MLA_CACHE_BF16)
      e = launch_attn_paged_bf16(p, grid, stream);
    else if (fmt == MLA_CACHE_FP8)
      e = launch_attn_paged_fp8(p, grid, stream);
    else
      e = launch_attn_paged_ds(p, grid, stream);
    prof_end(stream);
  }
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "decode attention launch failed: %s", cudaGetErrorString(e));
  if (sp.n_splits > 1) {
    MergeParams m{};
    m.part_o = part_o;
    m.part_lse = part_lse;
    m.S = sp.n_splits;
    m.n_rows = static_cast<int>(n_rows);
    m.H = H;
    m.seq_lens = seq_lens;
    m.q_len = q_len;
    m.chunk = sp.chunk;
    m.out = static_cast<uint8_t*>(out);
    m.o_s0b = o_s0 * 2;
    m.o_s1b = o_s1 * 2;
    m.lse = lse;
    if (launch_merge(m, stream) != cudaSuccess)
      return fail(MLA_ERR_CUDA, "merge launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  }
  return ok();
}

// ------------------------------------------------------------------------------------------
extern "C" int mla_gather_dequant(const void* kv_cache, mla_cache_format fmt, int64_t num_blocks,
                                  int64_t block_stride_bytes, int64_t entry_stride_bytes,
                                  int32_t block_size, const int64_t* slots, int64_t n, float* out,
                                  cudaStream_t stream) {
  if (fmt != MLA_CACHE_BF16 && fmt != MLA_CACHE_FP8 && fmt != MLA_CACHE_FP8_DS_MLA)
    return fail(MLA_ERR_INVALID, "unknown cache format %d", static_cast<int>(fmt));
  if (n < 0) return fail(MLA_ERR_INVALID, "n must be >= 0");
  if (n == 0) return ok();
  if (!kv_cache || !slots || !out) return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (block_size < 1 || num_blocks < 1 || entry_stride_bytes < entry_bytes(fmt) ||
      block_stride_bytes < entry_stride_bytes * block_size)
    return fail(MLA_ERR_INVALID, "bad cache geometry");
  if (fmt != MLA_CACHE_FP8 && (entry_stride_bytes % 4 || block_stride_bytes % 4 || !aligned(kv_cache, 4)))
    return fail(MLA_ERR_INVALID, "bf16 / fp8_ds_mla entries must be 4-byte aligned");
  if (n > (int64_t(1) << 33)) return fail(MLA_ERR_UNSUPPORTED, "n too large");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  GatherParams p{};
  p.cache = static_cast<const uint8_t*>(kv_cache);
  p.num_blocks = num_blocks;
  p.block_stride = block_stride_bytes;
  p.entry_stride = entry_stride_bytes;
  p.block_size = block_size;
  p.slots = slots;
  p.n = n;
  p.out = out;
  p.err = d->err;
  if (launch_gather(static_cast<int>(fmt), p, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "gather launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

// ------------------------------------------------------------------------------------------
extern "C" int mla_gather_context(const void* kv_cache, mla_cache_format fmt, int64_t num_blocks,
                                  int64_t block_stride_bytes, int64_t entry_stride_bytes, int32_t block_size,
                                  const int32_t* block_table, int64_t bt_stride, const int32_t* cu_seq_lens,
                                  const int32_t* seq_starts, int32_t batch, int64_t num_tokens, int32_t out_kind,
                                  float scale, void* dst, int64_t dst_row_stride_bytes, cudaStream_t stream) {
  if (fmt != MLA_CACHE_BF16 && fmt != MLA_CACHE_FP8 && fmt != MLA_CACHE_FP8_DS_MLA)
    return fail(MLA_ERR_INVALID, "unknown cache format %d", static_cast<int>(fmt));
  if (out_kind != MLA_GATHER_BF16 && out_kind != MLA_GATHER_RAW)
    return fail(MLA_ERR_INVALID, "unknown gather output kind %d", out_kind);
  if (batch < 0 || num_tokens < 0) return fail(MLA_ERR_INVALID, "batch and num_tokens must be >= 0");
  if (batch == 0 || num_tokens == 0) return ok();
  if (!kv_cache || !block_table || !cu_seq_lens || !dst) return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (block_size < 1 || num_blocks < 1 || bt_stride < 1 || entry_stride_bytes < entry_bytes(fmt) ||
      block_stride_bytes < entry_stride_bytes * block_size)
    return fail(MLA_ERR_INVALID, "bad cache geometry");
  const int64_t row_bytes = out_kind == MLA_GATHER_RAW ? entry_bytes(fmt) : 1152;
  if (dst_row_stride_bytes < row_bytes) return fail(MLA_ERR_INVALID, "dst rows overlap");
  if (out_kind == MLA_GATHER_BF16 && (!aligned(dst, 2) || dst_row_stride_bytes % 2))
    return fail(MLA_ERR_INVALID, "bf16 dst rows must be 2-byte aligned");
  if (fmt == MLA_CACHE_FP8_DS_MLA && (entry_stride_bytes % 4 || block_stride_bytes % 4 || !aligned(kv_cache, 4)))
    return fail(MLA_ERR_INVALID, "fp8_ds_mla entries must be 4-byte aligned");
  if (fmt == MLA_CACHE_BF16 && (entry_stride_bytes % 2 || block_stride_bytes % 2 || !aligned(kv_cache, 2)))
    return fail(MLA_ERR_INVALID, "bf16 entries must be 2-byte aligned");
  if (num_tokens >= (int64_t(1) << 33)) return fail(MLA_ERR_UNSUPPORTED, "num_tokens too large");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  GatherCtxParams p{};
  p.cache = static_cast<const uint8_t*>(kv_cache);
  p.num_blocks = num_blocks;
  p.block_stride = block_stride_bytes;
  p.entry_stride = entry_stride_bytes;
  p.block_size = block_size;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.cu = cu_seq_lens;
  p.starts = seq_starts;
  p.batch = batch;
  p.num_tokens = num_tokens;
  p.scale = scale;
  p.dst = static_cast<uint8_t*>(dst);
  p.dst_row = dst_row_stride_bytes;
  p.vec = aligned(kv_cache, 16) && entry_stride_bytes % 16 == 0 && block_stride_bytes % 16 == 0 && aligned(dst, 16) &&
          dst_row_stride_bytes % 16 == 0;
  p.err = d->err;
  if (launch_gather_context(static_cast<int>(fmt), out_kind, p, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "gather launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

extern "C" int mla_merge_attn_states(void* output, int64_t o_s0, int64_t o_s1, float* output_lse,
                                     const void* prefix_output, int64_t p_s0, int64_t p_s1, const float* prefix_lse,
                                     const void* suffix_output, int64_t s_s0, int64_t s_s1, const float* suffix_lse,
                                     int32_t T, int32_t H, int32_t D, cudaStream_t stream) {
  if (T < 0 || H < 1 || D < 1) return fail(MLA_ERR_INVALID, "bad shape T=%d H=%d D=%d", T, H, D);
  if (T == 0) return ok();
  if (!output || !prefix_output || !prefix_lse || !suffix_output || !suffix_lse)
    return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (o_s1 < D || o_s0 < static_cast<int64_t>(H) * o_s1 || p_s1 < D || p_s0 < static_cast<int64_t>(H) * p_s1 ||
      s_s1 < D || s_s0 < static_cast<int64_t>(H) * s_s1)
    return fail(MLA_ERR_INVALID, "strides overlap rows");
  if (!aligned(output, 2) || !aligned(prefix_output, 2) || !aligned(suffix_output, 2) || !aligned(prefix_lse, 4) ||
      !aligned(suffix_lse, 4) || (output_lse && !aligned(output_lse, 4)))
    return fail(MLA_ERR_INVALID, "misaligned tensor");
  MergeStatesParams p{};
  p.out = static_cast<uint16_t*>(output);
  p.o_s0 = o_s0;
  p.o_s1 = o_s1;
  p.out_lse = output_lse;
  p.prefix = static_cast<const uint16_t*>(prefix_output);
  p.p_s0 = p_s0;
  p.p_s1 = p_s1;
  p.prefix_lse = prefix_lse;
  p.suffix = static_cast<const uint16_t*>(suffix_output);
  p.s_s0 = s_s0;
  p.s_s1 = s_s1;
  p.suffix_lse = suffix_lse;
  p.T = T;
  p.H = H;
  p.D = D;
  p.vec = D % 8 == 0 && aligned(output, 16) && aligned(prefix_output, 16) && aligned(suffix_output, 16) &&
          o_s0 % 8 == 0 && o_s1 % 8 == 0 && p_s0 % 8 == 0 && p_s1 % 8 == 0 && s_s0 % 8 == 0 && s_s1 % 8 == 0;
  if (launch_merge_states(p, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "merge launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

// ------------------------------------------------------------------------------------------
// Per-head contractions around the attention core.
static int head_bmm(const void* x, int64_t x_s0, int64_t x_s1, const void* w, const void* gate, int64_t g_s0, void* y,
                    int64_t y_s0, int64_t y_s1, int32_t B, int32_t H, int32_t K, int32_t F, cudaStream_t stream) {
  if (B < 0 || H < 1) return fail(MLA_ERR_INVALID, "bad shape B=%d H=%d", B, H);
  if (K < 64 || K > 512 || K % 64) return fail(MLA_ERR_UNSUPPORTED, "the contraction length must be 64..512 in steps of 64, got %d", K);
  if (F < 128 || F % 128) return fail(MLA_ERR_UNSUPPORTED, "the output width must be a multiple of 128, got %d", F);
  if (B == 0) return ok();
  if (!x || !w || !y) return fail(MLA_ERR_INVALID, "a required pointer is NULL");
  if (x_s1 < K || x_s0 < static_cast<int64_t>(H) * x_s1 || y_s1 < F || y_s0 < static_cast<int64_t>(H) * y_s1 ||
      (gate && g_s0 < static_cast<int64_t>(H) * F))
    return fail(MLA_ERR_INVALID, "strides overlap rows");
  if (!aligned(w, 16) || !aligned(x, 2) || !aligned(y, 2) || (gate && !aligned(gate, 2)))
    return fail(MLA_ERR_INVALID, "the weights must be 16-byte aligned, bf16 tensors 2-byte aligned");
  if (static_cast<int64_t>(H) > 65535 || (static_cast<int64_t>(B) + 63) / 64 > 65535)
    return fail(MLA_ERR_UNSUPPORTED, "grid too large");
  DevInfo* d = nullptr;
  if (int rc = dev_info(&d)) return rc;
  HeadBmmParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.x_s0 = x_s0;
  p.x_s1 = x_s1;
  p.w = static_cast<const uint16_t*>(w);
  p.gate = static_cast<const uint16_t*>(gate);
  p.g_s0 = g_s0;
  p.y = static_cast<uint16_t*>(y);
  p.y_s0 = y_s0;
  p.y_s1 = y_s1;
  p.B = B;
  p.H = H;
  p.K = K;
  p.F = F;
  p.vec = aligned(x, 16) && x_s0 % 8 == 0 && x_s1 % 8 == 0;
  p.err = d->err;
  if (launch_head_bmm(p, stream) != cudaSuccess)
    return fail(MLA_ERR_CUDA, "per-head contraction launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return ok();
}

extern "C" int mla_absorb_q(const void* q_nope, int64_t qn_s0, int64_t qn_s1, const void* w_uk_t, void* ql_nope,
                            int64_t ql_s0, int64_t ql_s1, int32_t B, int32_t H, int32_t P, cudaStream_t stream) {
  return head_bmm(q_nope, qn_s0, qn_s1, w_uk_t, nullptr, 0, ql_nope, ql_s0, ql_s1, B, H, P, kLora, stream);
}

extern "C" int mla_v_up_proj(const void* latent, int64_t l_s0, int64_t l_s1, const void* w_uv, const void* gate,
                             int64_t g_s0, void* out, int64_t o_s0, int64_t o_s1, int32_t B, int32_t H, int32_t V,
                             cudaStream_t stream) {
  return head_bmm(latent, l_s0, l_s1, w_uv, gate, g_s0, out, o_s0, o_s1, B, H, kLora, V, stream);
}
