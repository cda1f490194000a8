// fp8_ds_mla attention kernel instantiations: sparse (gather warps) and paged (TMA pages).
#include "mla_ds.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

template <bool kSparse, int kCl>
cudaError_t configure(int dev) {
  static bool configured[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(mla_ds_kernel<kSparse, kCl>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, DsCfg<kSparse>::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return cudaSuccess;
}

template <bool kSparse>
cudaError_t launch_t(const DsParams& p, const void* tkv, const void* tsc, int grid, cudaStream_t stream) {
  using C = DsCfg<kSparse>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = configure<kSparse, 1>(dev)) != cudaSuccess) return e;
  CUtensorMap dummy{};
  const CUtensorMap& a = tkv ? *static_cast<const CUtensorMap*>(tkv) : dummy;
  const CUtensorMap& b = tsc ? *static_cast<const CUtensorMap*>(tsc) : dummy;
  return launch_pdl(mla_ds_kernel<kSparse, 1>, dim3(grid), dim3(C::kThreads), C::kAlloc, stream, p, a, b);
}

template <int kCl>
cudaLaunchAttribute cluster_attr() {
  cudaLaunchAttribute a{};
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = kCl;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

template <int kCl>
int capacity_t() {
  static int cap[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cap[dev] > 0) return cap[dev];
  if (configure<false, kCl>(dev) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kCl);
  cfg.blockDim = dim3(DsCfg<false>::kThreads);
  cfg.dynamicSmemBytes = DsCfg<false>::kAlloc;
  cudaLaunchAttribute attr[1] = {cluster_attr<kCl>()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_ds_kernel<false, kCl>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cap[dev] = n;
  return n;
}

template <int kCl>
cudaError_t launch_cl(const DsParams& p, const void* tkv, const void* tsc, int clusters, cudaStream_t stream) {
  using C = DsCfg<false>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = configure<false, kCl>(dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kCl * clusters);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2] = {cluster_attr<kCl>(), {}};
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mla_ds_kernel<false, kCl>, p, *static_cast<const CUtensorMap*>(tkv),
                            *static_cast<const CUtensorMap*>(tsc));
}

}  // namespace

// How many clusters of `size` CTAs (2, 3 or 6) of the paged kernel can be resident at once on
// this device (0 when the query fails or the size is not built): the persistent grid must not
// exceed it.
int ds_cluster_capacity(int size) {
  switch (size) {
    case 2:
      return capacity_t<2>();
    case 3:
      return capacity_t<3>();
    case 6:
      return capacity_t<6>();
    default:
      return 0;
  }
}

cudaError_t launch_ds_sparse(const DsParams& p, int grid, cudaStream_t stream) {
  return launch_t<true>(p, nullptr, nullptr, grid, stream);
}
cudaError_t launch_ds_paged(const DsParams& p, const void* tkv, const void* tsc, int grid, cudaStream_t stream) {
  return launch_t<false>(p, tkv, tsc, grid, stream);
}

// The paged kernel as CTA pairs: `pairs` 2-CTA clusters, p.n_items counting pair items.
// The paged kernel as clusters of `size` CTAs: `clusters` clusters, p.n_items counting
// cluster items.
cudaError_t launch_ds_paged_clusters(const DsParams& p, const void* tkv, const void* tsc, int size, int clusters,
                                     cudaStream_t stream) {
  switch (size) {
    case 2:
      return launch_cl<2>(p, tkv, tsc, clusters, stream);
    case 3:
      return launch_cl<3>(p, tkv, tsc, clusters, stream);
    case 6:
      return launch_cl<6>(p, tkv, tsc, clusters, stream);
    default:
      return cudaErrorInvalidValue;
  }
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
