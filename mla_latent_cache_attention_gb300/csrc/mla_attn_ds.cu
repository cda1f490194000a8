// Attention instantiations over fp8_ds_mla records: sparse (CSR) forward and paged decode.
#include "mla_attn_launch.cuh"
namespace mla {
cudaError_t launch_attn_sparse_ds(const AttnParams& p, int grid, cudaStream_t s) { return launch_attn<kDS, true>(p, grid, s); }
cudaError_t launch_attn_paged_ds(const AttnParams& p, int grid, cudaStream_t s) { return launch_attn<kDS, false>(p, grid, s); }
}  // namespace mla
