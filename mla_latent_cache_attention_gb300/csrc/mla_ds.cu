// fp8_ds_mla attention kernel instantiations: sparse (gather warps) and paged (TMA pages).
#include "mla_ds.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

template <bool kSparse>
cudaError_t launch_t(const DsParams& p, const void* tkv, const void* tsc, int grid, cudaStream_t stream) {
  using C = DsCfg<kSparse>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(mla_ds_kernel<kSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  CUtensorMap dummy{};
  const CUtensorMap& a = tkv ? *static_cast<const CUtensorMap*>(tkv) : dummy;
  const CUtensorMap& b = tsc ? *static_cast<const CUtensorMap*>(tsc) : dummy;
  return launch_pdl(mla_ds_kernel<kSparse>, dim3(grid), dim3(C::kThreads), C::kAlloc, stream, p, a, b);
}

}  // namespace

cudaError_t launch_ds_sparse(const DsParams& p, int grid, cudaStream_t stream) {
  return launch_t<true>(p, nullptr, nullptr, grid, stream);
}
cudaError_t launch_ds_paged(const DsParams& p, const void* tkv, const void* tsc, int grid, cudaStream_t stream) {
  return launch_t<false>(p, tkv, tsc, grid, stream);
}

}  // namespace mla

#ifdef MLA_TIMELINE
extern "C" __attribute__((visibility("default"))) int mla_debug_timeline_ds(void* events, void* counts) {
  cudaMemcpyFromSymbol(events, mla::g_tl, sizeof(mla::g_tl));
  cudaMemcpyFromSymbol(counts, mla::g_tl_n, sizeof(mla::g_tl_n));
  const int zero[mla::kTlCtas][mla::kTlRoles] = {};
  return cudaMemcpyToSymbol(mla::g_tl_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -3;
}
#endif
