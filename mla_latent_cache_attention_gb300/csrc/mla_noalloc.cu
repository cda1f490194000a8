// mla_noalloc.cu -- paged decode for callers that cannot allocate device memory.
//
// mla_paged_decode needs a caller-provided workspace for its split-K partials.  Some callers
// cannot produce one: code that runs inside a region where cudaMalloc is not allowed (for
// instance while a CUDA stream is being captured, where an allocation would break the
// capture), plug-ins embedded in an engine that owns every byte of device memory through its
// own pool and hands none to the plug-in, and latency-critical serving loops that forbid
// allocation on the request path.  mla_paged_decode_noalloc serves them with a scratch
// buffer that lives in the library itself: a file-scope __device__ array of
// kNoAllocScratchBytes (64 MiB).  The call allocates nothing.
//
// The scratch is shared by every call in the process on that device and keeps the previous
// call's contents; the decode writes every partial it later reads, so nothing has to be
// cleared between calls.  Two calls whose kernels overlap on the GPU (different streams
// without ordering between them) race on the scratch and give wrong results.
#include <cstdio>
#include <mutex>

#include "mla.h"
#include "mla_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchSlot {
  bool ready = false;
  void* ptr = nullptr;
};
ScratchSlot g_scratch[64];
std::mutex g_scratch_mu;

// Device address of the scratch on the current device (set up once per device).  In host
// code g_noalloc_scratch names a host-side stand-in, so the address must come from
// cudaGetSymbolAddress with that device current.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    mla::set_error_message("mla_paged_decode_noalloc: cudaGetDevice failed");
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchSlot& s = g_scratch[dev];
  if (!s.ready) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof msg,
               "mla_paged_decode_noalloc: cudaGetSymbolAddress of the static scratch failed on device %d: %s",
               dev, cudaGetErrorString(e));
      mla::set_error_message(msg);
      return MLA_ERR_CUDA;
    }
    s.ptr = p;
    s.ready = true;
  }
  *out = s.ptr;
  return MLA_OK;
}

}  // namespace

extern "C" int mla_paged_decode_noalloc(const void* q, int64_t q_s0, int64_t q_s1, const void* kv_cache,
                                        mla_cache_format fmt, int64_t num_blocks, int64_t block_stride_bytes,
                                        int64_t entry_stride_bytes, int32_t block_size,
                                        const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                                        int32_t B, int32_t q_len, int32_t H, int32_t max_context,
                                        float softmax_scale, float q_scale, float k_scale, void* out,
                                        int64_t o_s0, int64_t o_s1, float* lse, cudaStream_t stream) {
  if (B > 0 && q_len > 0 && H > 0 && max_context > 0) {
    const size_t need = mla_paged_decode_workspace_size(B, q_len, H, max_context, 0);
    if (need > kNoAllocScratchBytes) {
      char msg[256];
      snprintf(msg, sizeof msg,
               "mla_paged_decode_noalloc: this shape needs %zu bytes of split-K scratch; the library's static "
               "scratch holds %zu bytes (use mla_paged_decode with a caller workspace)",
               need, kNoAllocScratchBytes);
      mla::set_error_message(msg);
      return MLA_ERR_UNSUPPORTED;
    }
  }
  void* scratch = nullptr;
  if (int rc = scratch_on_current_device(&scratch)) return rc;
  return mla_paged_decode(q, q_s0, q_s1, kv_cache, fmt, num_blocks, block_stride_bytes, entry_stride_bytes,
                          block_size, block_table, bt_stride, seq_lens, B, q_len, H, max_context, softmax_scale,
                          q_scale, k_scale, out, o_s0, o_s1, lse, scratch, kNoAllocScratchBytes, stream);
}
