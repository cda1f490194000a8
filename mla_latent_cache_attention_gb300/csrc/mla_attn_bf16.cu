// Attention instantiation: paged decode over the bf16 cache.
#include "mla_attn_launch.cuh"
namespace mla {
cudaError_t launch_attn_paged_bf16(const AttnParams& p, int grid, cudaStream_t s) { return launch_attn<kBF16, false>(p, grid, s); }
}  // namespace mla

#ifdef MLA_TIMELINE
extern "C" __attribute__((visibility("default"))) int mla_debug_timeline(void* events, void* counts) {
  cudaMemcpyFromSymbol(events, mla::g_tl, sizeof(mla::g_tl));
  cudaMemcpyFromSymbol(counts, mla::g_tl_n, sizeof(mla::g_tl_n));
  const int zero[mla::kTlCtas][mla::kTlRoles] = {};
  return cudaMemcpyToSymbol(mla::g_tl_n, zero, sizeof(zero)) == cudaSuccess ? 0 : -3;
}
#endif
