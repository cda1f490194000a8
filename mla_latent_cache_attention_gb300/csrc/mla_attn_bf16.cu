// Attention instantiation: paged decode over the bf16 cache.
#include "mla_attn_launch.cuh"
namespace mla {
cudaError_t launch_attn_paged_bf16(const AttnParams& p, int grid, cudaStream_t s) { return launch_attn<kBF16, false>(p, grid, s); }
}  // namespace mla

