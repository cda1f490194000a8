// Attention instantiation: paged decode / spec-verify over the plain fp8 cache.
#include "mla_attn_launch.cuh"
namespace mla {
cudaError_t launch_attn_paged_fp8(const AttnParams& p, int grid, cudaStream_t s) { return launch_attn<kFP8, false>(p, grid, s); }
}  // namespace mla
