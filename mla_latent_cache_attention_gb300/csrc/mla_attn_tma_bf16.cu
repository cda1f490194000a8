// Attention instantiation: paged decode over the bf16 cache with TMA page loads.
#include "mla_attn_tma.cuh"
#include "mla_internal.h"

namespace mla {

cudaError_t launch_attn_tma_bf16(const AttnParams& p, const void* tmap, int grid, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(mla_attn_tma_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TmaSmem::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  mla_attn_tma_bf16_kernel<<<grid, kTmaThreads, TmaSmem::kAlloc, stream>>>(p, *static_cast<const CUtensorMap*>(tmap));
  return cudaGetLastError();
}

}  // namespace mla

#ifdef MLA_TIMELINE
extern "C" __attribute__((visibility("default"))) int mla_debug_timeline(void* events, void* counts) {
  cudaMemcpyFromSymbol(events, mla::g_tl, sizeof(mla::g_tl));
  cudaMemcpyFromSymbol(counts, mla::g_tl_n, sizeof(mla::g_tl_n));
  const int zero[mla::kTlCtas][mla::kTlRoles] = {};
  return cudaMemcpyToSymbol(mla::g_tl_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -3;
}
#endif
