// mla_head_bmm.cu -- the per-head contractions around the attention core of the absorbed MLA
// decode, on the tcgen05 tensor cores:
//   BMM1   ql_nope[b, h, :] = q_nope[b, h, :] . W_UK_T[h]        (K = qk_nope_head_dim, F = 512)
//   W_UV   out[b, h, :]     = latent[b, h, :] . W_UV[h]           (K = 512, F = v_head_dim)
//          optionally times bf16(sigmoid(gate[b, h * F + f]))    (the output gate)
// "vllm.models.kimi_k3.nvidia.mla": _attention (BMM1), _v_up_proj and the gate of forward.
//
// One CTA per (head, 128 output features, 64 tokens): the weight tile [K x 128 features] is
// the MN-major A operand (M = features, two 64-wide SW128 halves), the tokens' K values the
// K-major B operand (N = 64), the fp32 accumulator D[128 x 64] lives in TMEM.  Operands are
// staged with 16-byte loads straight into the swizzled layouts; one thread issues the K / 16
// MMAs; four warps read D back (lane = feature, column = token) and write bf16 rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "mla_ptx.cuh"

namespace mla {
namespace {

constexpr int kHbN = 64;          // tokens per CTA (MMA N)
constexpr int kHbThreads = 128;

__device__ __forceinline__ uint32_t swz(int row, int c) {
  return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

__global__ void __launch_bounds__(kHbThreads, 1) mla_head_bmm_kernel(const HeadBmmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int K = p.K, F = p.F;
  uint8_t* sa = smem;                          // 2 halves x [K rows x 128 B]
  uint8_t* sb = smem + 256 * K;                // K / 64 blocks x [64 tokens x 128 B]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 384 * K);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 384 * K + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 384 * K + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, f0 = blockIdx.y * 128, b0 = blockIdx.z * kHbN;

  if (tid == 0) {
    mbar_init(bar, 1);
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kHbN);
    tmem_relinquish();
  }
  // weight tile: row k holds features f0 .. f0 + 127 (256 bytes = 16 chunks of 8)
  const uint16_t* wh = p.w + static_cast<int64_t>(h) * K * F + f0;
  for (int i = tid; i < K * 16; i += kHbThreads) {
    const int k = i >> 4, c = i & 15;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(wh + static_cast<int64_t>(k) * F + 8 * c));
    *reinterpret_cast<uint4*>(sa + (c >> 3) * (K * 128) + swz(k, c & 7)) = v;
  }
  // token rows: K / 8 chunks of 8 values each; tokens past B are zero
  const int kc = K >> 3;
  for (int i = tid; i < kHbN * kc; i += kHbThreads) {
    const int n = i / kc, c = i - n * kc, b = b0 + n;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (b < p.B) {
      const uint16_t* src = p.x + b * p.x_s0 + h * p.x_s1 + 8 * c;
      if (p.vec) {
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        uint16_t e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) e[u] = src[u];
        v = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
      }
    }
    *reinterpret_cast<uint4*>(sb + (c >> 3) * (kHbN * 128) + swz(n, c & 7)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    const uint64_t da = smem_desc(smem_u32(sa), K * 128, 1024, kSwizzle128B);   // MN-major: LBO = next 64 features
    const uint64_t db = smem_desc(smem_u32(sb), 16, 1024, kSwizzle128B);        // K-major
    constexpr uint32_t kId = idesc_f16(128, kHbN, 1, 1, 1, 0);
    for (int s = 0; s < K / 16; ++s)
      mma_f16_ss(tmem, da + ((s * 2048) >> 4), db + (((s >> 2) * (kHbN * 128) + (s & 3) * 32) >> 4), kId,
                 s > 0 ? 1u : 0u);
    mma_commit(bar);
  }
  __syncwarp();
  const bool ok = mbar_wait(bar, 0, abort_flag);
  tc_fence_after();
  // epilogue: lane = feature f0 + 32 warp + lane, 16 token columns per TMEM load
  const int f = f0 + 32 * warp + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  if (ok) {
#pragma unroll 1
    for (int j = 0; j < kHbN / 16; ++j) {
      float v[16];
      tmem_ld16(tl + 16 * j, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int b = b0 + 16 * j + i;
        if (b >= p.B) break;
        uint16_t y = to_bf16_bits(v[i]);
        if (p.gate) {
          const float g = __uint_as_float(static_cast<uint32_t>(p.gate[b * p.g_s0 + static_cast<int64_t>(h) * F + f]) << 16);
          const float sg = __uint_as_float(static_cast<uint32_t>(to_bf16_bits(1.f / (1.f + __expf(-g)))) << 16);
          y = to_bf16_bits(__uint_as_float(static_cast<uint32_t>(y) << 16) * sg);
        }
        p.y[b * p.y_s0 + h * p.y_s1 + f] = y;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag == 2) set_device_error(p.err, 16u);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kHbN);
  }
}

}  // namespace

int head_bmm_smem_bytes(int K) { return 384 * K + 64 + 1024; }

cudaError_t launch_head_bmm(const HeadBmmParams& p, cudaStream_t stream) {
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int smem = head_bmm_smem_bytes(p.K);
  if (configured[dev] < smem) {
    e = cudaFuncSetAttribute(mla_head_bmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, head_bmm_smem_bytes(512));
    if (e != cudaSuccess) return e;
    configured[dev] = head_bmm_smem_bytes(512);
  }
  const dim3 grid(p.H, p.F / 128, (p.B + kHbN - 1) / kHbN);
  mla_head_bmm_kernel<<<grid, kHbThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
