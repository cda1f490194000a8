// Paged decode kernel instantiations for the bf16 cache (TMA page loads, ring pipeline).
#include "mla_internal.h"
#include "mla_paged_tma.cuh"

namespace mla {
namespace {

template <int NQ>
cudaError_t launch_nq(const PagedParams& p, const void* tkv, const void* tq, int grid, cudaStream_t stream) {
  using C = PagedCfg<kBF16, NQ>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(mla_paged_tma_kernel<kBF16, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_pdl(mla_paged_tma_kernel<kBF16, NQ>, dim3(grid), dim3(C::kThreads), C::kAlloc, stream, p,
                    *static_cast<const CUtensorMap*>(tkv), *static_cast<const CUtensorMap*>(tq));
}

}  // namespace

cudaError_t launch_paged_tma_bf16(int nq, const PagedParams& p, const void* tkv, const void* tq, int grid,
                                 cudaStream_t stream) {
  switch (nq) {
    case 16:
      return launch_nq<16>(p, tkv, tq, grid, stream);
    case 32:
      return launch_nq<32>(p, tkv, tq, grid, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace mla

#ifdef MLA_TIMELINE
extern "C" __attribute__((visibility("default"))) int mla_debug_timeline_bf16(void* events, void* counts) {
  cudaMemcpyFromSymbol(events, mla::g_tl, sizeof(mla::g_tl));
  cudaMemcpyFromSymbol(counts, mla::g_tl_n, sizeof(mla::g_tl_n));
  const int zero[mla::kTlCtas][mla::kTlRoles] = {};
  return cudaMemcpyToSymbol(mla::g_tl_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -3;
}
#endif
