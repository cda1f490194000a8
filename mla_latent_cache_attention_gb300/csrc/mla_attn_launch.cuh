// mla_attn_launch.cuh -- host launcher of one attention kernel instantiation.
#pragma once
#include "mla_attn.cuh"
#include "mla_internal.h"

namespace mla {

template <int F, bool kSparse>
cudaError_t launch_attn(const AttnParams& p, int grid, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(mla_attn_kernel<F, kSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<F>::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_pdl(mla_attn_kernel<F, kSparse>, dim3(grid), dim3(kThreads), Smem<F>::kAlloc, stream, p);
}

}  // namespace mla
