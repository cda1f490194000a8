// mla_small_kernels.cu -- the memory-bound kernels around the attention core:
//   * the decode epilogue (q concat + latent insert), one CTA per (token, 4 heads) and one
//     per token for the insert;
//   * the split-K merge of partial attentions by their log-sum-exp;
//   * gather-and-dequantise of cache entries (a test aid with the kernels' addressing).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "mla_ptx.cuh"

namespace mla {

// ------------------------------------------------------------------------------------------
// Decode epilogue.  "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache",
// fused_mla_decode_q_concat_kv_cache_insert: mqa_q = [ql_nope | q_pe], then the latent
// [kv_c_normed | k_pe] is written at slot_mapping; optional GPT-J RoPE from an fp32 table.

__device__ __forceinline__ float bf16_at(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(*p) << 16);
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}
__device__ __forceinline__ uint8_t e4m3_sat(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// GPT-J rotation of pair (x0, x1) by (c, s) in fp32: y0 = x0*c - x1*s, y1 = x1*c + x0*s with
// the product x1*s (x0*s) rounded before the fused multiply-add.
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& y0, float& y1) {
  y0 = __fmaf_rn(x0, c, -__fmul_rn(x1, s));
  y1 = __fmaf_rn(x1, c, __fmul_rn(x0, s));
}

// fp8_ds_mla tile scale: 2^k with k the least integer such that amax <= 448 * 2^k,
// clamped to k >= -126; an all-zero tile gets k = 0.  Works on the fp32 bits of amax
// (448 * 2^k = 1.75 * 2^(8+k)).
__device__ __forceinline__ int ds_tile_exponent(float amax) {
  const uint32_t u = __float_as_uint(amax);
  if (u == 0u) return 0;
  const int e_field = static_cast<int>(u >> 23);
  if (e_field == 0) return -126;                       // subnormal amax
  const int E = e_field - 127;
  const uint32_t m = u & 0x7FFFFFu;
  int k = E - 8 + (m > 0x600000u ? 1 : 0);
  return k < -126 ? -126 : k;
}

// Write one cache entry (128 threads): [kv_c | rope(k_pe)] as bf16 (F = 0), as
// e4m3_sat(x * cinv) (F = 1), or as a 656-byte fp8_ds_mla record (F = 2: per-128-tile scale
// 2^k from ds_tile_exponent, codes e4m3(x / 2^k), rope bf16).  cs: the RoPE row or null.
template <int F>
__device__ __forceinline__ void insert_latent(uint8_t* ent, const uint16_t* __restrict__ kc,
                                              const uint16_t* __restrict__ kr, const float* __restrict__ cs, float cinv,
                                              int tid) {
  if (tid < 32) {   // rope part, one pair per lane
    float y0 = bf16_at(kr + 2 * tid), y1 = bf16_at(kr + 2 * tid + 1);
    if (cs) rope_pair(y0, y1, cs[tid], cs[32 + tid], y0, y1);
    if (F == 0) {
      reinterpret_cast<uint16_t*>(ent)[512 + 2 * tid] = bf16_bits(y0);
      reinterpret_cast<uint16_t*>(ent)[512 + 2 * tid + 1] = bf16_bits(y1);
    } else if (F == 1) {
      ent[512 + 2 * tid] = e4m3_sat(y0 * cinv);
      ent[512 + 2 * tid + 1] = e4m3_sat(y1 * cinv);
    } else {
      reinterpret_cast<uint16_t*>(ent + 528)[2 * tid] = bf16_bits(y0);
      reinterpret_cast<uint16_t*>(ent + 528)[2 * tid + 1] = bf16_bits(y1);
    }
  }
  // NoPE part: warp w owns the 128-wide tile w, 4 values per lane
  const int w = tid >> 5, lane = tid & 31;
  float x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = bf16_at(kc + 128 * w + 4 * lane + i);
  if (F == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) reinterpret_cast<uint16_t*>(ent)[128 * w + 4 * lane + i] = kc[128 * w + 4 * lane + i];
  } else if (F == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) ent[128 * w + 4 * lane + i] = e4m3_sat(x[i] * cinv);
  } else {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int k = ds_tile_exponent(amax);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);   // 2^-k, exact
#pragma unroll
    for (int i = 0; i < 4; ++i) ent[128 * w + 4 * lane + i] = e4m3_sat(x[i] * inv);
    if (lane == 0) {
      const float s = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
      *reinterpret_cast<float*>(ent + 512 + 4 * w) = s;
    }
  }
}

// Grid (B, ceil(H / 4) + 1): CTA (b, g < ceil(H / 4)) builds the query rows of heads
// 4g..4g+3 of token b; CTA (b, ceil(H / 4)) inserts token b's latent, in parallel with them.
// Loads go through restrict-qualified pointers in batches of 8 so that they are all in
// flight before the stores.
template <int F>
__global__ void __launch_bounds__(128) mla_epilogue_kernel(const EpiParams p) {
  const int b = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  // the decode launched next (a programmatic dependent) may be scheduled now; it waits for
  // this grid before it reads the query and the cache
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const bool inserter = g == static_cast<int>(gridDim.y) - 1;
  const int64_t slot = inserter ? p.slot_mapping[b] : -1;     // loaded with the position
  const float qinv = (F == 1) ? *p.q_scale_inv : 1.f;
  const float cinv = (F == 1) ? *p.cache_scale_inv : 1.f;
  const float* __restrict__ cs = nullptr;
  if (p.positions) {
    int64_t pos = p.positions[b];
    if (pos < 0 || pos >= p.max_position) {
      if (tid == 0 && inserter) set_device_error(p.err, 8u);
      pos = pos < 0 ? 0 : p.max_position - 1;
    }
    cs = p.cos_sin + pos * 64;
  }
  if (inserter) {
    // ---- latent insert
    if (slot < 0) return;
    const int64_t blk = slot / p.block_size;
    if (blk >= p.num_blocks) {
      if (tid == 0) set_device_error(p.err, 4u);
      return;
    }
    insert_latent<F>(p.cache + blk * p.block_stride + (slot % p.block_size) * p.entry_stride, p.kv_c + b * p.kv_s0,
                     p.k_pe + b * p.kp_s0, cs, cinv, tid);
    return;
  }
  const int H = p.H;
  const int h_lo = 4 * g, h_hi = min(H, 4 * g + 4);
  const uint16_t* __restrict__ qn = p.ql_nope;
  const uint16_t* __restrict__ qpe = p.q_pe;
  // ---- query concat: 64 groups of 8 NoPE values and 8 rope pairs per head
  for (int i = tid; i < (h_hi - h_lo) * 64; i += blockDim.x) {
    const int h = h_lo + (i >> 6), d0 = (i & 63) * 8;
    const uint16_t* src = qn + b * p.ql_s0 + h * p.ql_s1 + d0;
    const int64_t o = (static_cast<int64_t>(b) * H + h) * 576 + d0;
    uint16_t v[8];
    if (p.vec16) {       // 16-byte aligned rows: one vector load (and store for 16-bit outputs)
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
      if (F != 1) {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.mqa_q) + o) = w;
        continue;
      }
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[2 * e] = static_cast<uint16_t>(ww[e] & 0xFFFFu);
        v[2 * e + 1] = static_cast<uint16_t>(ww[e] >> 16);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = __ldg(src + e);
    }
    if (F == 1) {
      uint8_t* __restrict__ q8 = reinterpret_cast<uint8_t*>(p.mqa_q) + o;
#pragma unroll
      for (int e = 0; e < 8; ++e) q8[e] = e4m3_sat(__uint_as_float(static_cast<uint32_t>(v[e]) << 16) * qinv);
    } else {
      uint16_t* __restrict__ q16 = reinterpret_cast<uint16_t*>(p.mqa_q) + o;
#pragma unroll
      for (int e = 0; e < 8; ++e) q16[e] = v[e];
    }
  }
  for (int i = tid; i < (h_hi - h_lo) * 32; i += blockDim.x) {
    const int h = h_lo + (i >> 5), pr = i & 31;
    const uint16_t* src = qpe + b * p.qp_s0 + h * p.qp_s1 + 2 * pr;
    float y0 = bf16_at(src), y1 = bf16_at(src + 1);
    if (cs) rope_pair(y0, y1, cs[pr], cs[32 + pr], y0, y1);
    const int64_t o = (static_cast<int64_t>(b) * H + h) * 576 + 512 + 2 * pr;
    if (F == 1) {
      uint8_t* q8 = reinterpret_cast<uint8_t*>(p.mqa_q);
      q8[o] = e4m3_sat(y0 * qinv);
      q8[o + 1] = e4m3_sat(y1 * qinv);
    } else {
      uint16_t* q16 = reinterpret_cast<uint16_t*>(p.mqa_q);
      q16[o] = bf16_bits(y0);
      q16[o + 1] = bf16_bits(y1);
    }
  }
}

// ------------------------------------------------------------------------------------------
// Prefill epilogues.  "vllm.models.kimi_k3.nvidia.ops.fused_mla_key_concat_kv_cache":
//   F = 0 / 2  fused_mla_key_concat_kv_cache_insert / fused_mla_key_concat_ds_mla_insert:
//              k_out[t, h] = [k_nope[t, h] | rope(k_pe[t])] (bf16), the last 64 values of
//              q[t, h] rotated in place, the latent inserted into the bf16 / fp8_ds_mla cache;
//   F = 1      fused_mla_qkv_quant_kv_cache_fp8_insert: q / k / v quantised to E4M3 with their
//              own scales (q rotated on the way, not in place), the latent into the plain fp8
//              cache with the cache scale.
// Grid (Tp, ceil(H / 4)), 128 threads: CTA (t, g) handles heads 4g..4g+3 of token t and, for
// g == 0, the latent insert of token t.  rope(k_pe[t]) is formed once per CTA in shared memory.

// 8 consecutive bf16 values as fp32 (one 16-byte load when vec, else scalar loads)
__device__ __forceinline__ void load8(const uint16_t* __restrict__ src, bool vec, float (&x)[8]) {
  if (vec) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(ww[e] << 16);
      x[2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = bf16_at(src + e);
  }
}

// 8 values quantised with inv to E4M3 (one 8-byte store when vec)
__device__ __forceinline__ void store8_e4m3(uint8_t* dst, bool vec, const float (&x)[8], float inv) {
  uint8_t c[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) c[e] = e4m3_sat(x[e] * inv);
  if (vec) {
    uint2 w;
    w.x = c[0] | (c[1] << 8) | (c[2] << 16) | (static_cast<uint32_t>(c[3]) << 24);
    w.y = c[4] | (c[5] << 8) | (c[6] << 16) | (static_cast<uint32_t>(c[7]) << 24);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) dst[e] = c[e];
  }
}

template <int F>
__global__ void __launch_bounds__(128) mla_prefill_epilogue_kernel(const PrefillEpiParams p) {
  const int t = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  __shared__ float kpr[64];        // rope(k_pe[t]) in fp32
  const float* __restrict__ cs = nullptr;
  if (p.positions) {
    int64_t pos = p.positions[t];
    if (pos < 0 || pos >= p.max_position) {
      if (tid == 0 && g == 0) set_device_error(p.err, 8u);
      pos = pos < 0 ? 0 : p.max_position - 1;
    }
    cs = p.cos_sin + pos * 64;
  }
  const uint16_t* __restrict__ kr = p.k_pe + t * p.kp_s0;
  if (tid < 32) {
    float y0 = bf16_at(kr + 2 * tid), y1 = bf16_at(kr + 2 * tid + 1);
    if (cs) rope_pair(y0, y1, cs[tid], cs[32 + tid], y0, y1);
    kpr[2 * tid] = y0;
    kpr[2 * tid + 1] = y1;
  }
  __syncthreads();
  const float qinv = (F == 1) ? *p.q_scale_inv : 1.f;
  const float kinv = (F == 1) ? *p.k_scale_inv : 1.f;
  const float vinv = (F == 1) ? *p.v_scale_inv : 1.f;
  const int H = p.H, dn = p.dn, de = p.dn + 64;
  const bool vec = p.vec != 0;
  const int h_lo = 4 * g, h_hi = min(H, 4 * g + 4), nh = h_hi - h_lo;
  // ---- NoPE parts: 8 values per item (k_nope -> k_out / k8, and for fp8 q_nope -> q8, v -> v8)
  const int cn = dn >> 3;
  for (int i = tid; i < nh * cn; i += blockDim.x) {
    const int h = h_lo + i / cn, d0 = (i % cn) * 8;
    const int64_t o = (static_cast<int64_t>(t) * H + h) * de + d0;
    const uint16_t* kn = p.k_nope + t * p.kn_s0 + h * p.kn_s1 + d0;
    if (F == 1) {
      float x[8];
      load8(kn, vec, x);
      store8_e4m3(p.k8 + o, vec, x, kinv);
      load8(p.q + t * p.q_s0 + h * p.q_s1 + d0, vec, x);
      store8_e4m3(p.q8 + o, vec, x, qinv);
    } else if (vec) {
      *reinterpret_cast<uint4*>(p.k_out + o) = __ldg(reinterpret_cast<const uint4*>(kn));
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) p.k_out[o + e] = kn[e];
    }
  }
  if (F == 1) {
    const int cv = p.dv >> 3;
    for (int i = tid; i < nh * cv; i += blockDim.x) {
      const int h = h_lo + i / cv, d0 = (i % cv) * 8;
      float x[8];
      load8(p.v + t * p.v_s0 + h * p.v_s1 + d0, vec, x);
      store8_e4m3(p.v8 + (static_cast<int64_t>(t) * H + h) * p.dv + d0, vec, x, vinv);
    }
  }
  // ---- rope parts: one pair per item (q rotated, k_out / k8 from the shared rotation)
  for (int i = tid; i < nh * 32; i += blockDim.x) {
    const int h = h_lo + (i >> 5), pr = i & 31;
    const int64_t o = (static_cast<int64_t>(t) * H + h) * de + dn + 2 * pr;
    uint16_t* qp = p.q + t * p.q_s0 + h * p.q_s1 + dn + 2 * pr;
    float y0 = bf16_at(qp), y1 = bf16_at(qp + 1);
    if (cs) rope_pair(y0, y1, cs[pr], cs[32 + pr], y0, y1);
    if (F == 1) {
      p.q8[o] = e4m3_sat(y0 * qinv);
      p.q8[o + 1] = e4m3_sat(y1 * qinv);
      p.k8[o] = e4m3_sat(kpr[2 * pr] * kinv);
      p.k8[o + 1] = e4m3_sat(kpr[2 * pr + 1] * kinv);
    } else {
      if (cs) {
        qp[0] = bf16_bits(y0);
        qp[1] = bf16_bits(y1);
      }
      p.k_out[o] = bf16_bits(kpr[2 * pr]);
      p.k_out[o + 1] = bf16_bits(kpr[2 * pr + 1]);
    }
  }
  if (g != 0) return;
  // ---- latent insert
  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;
  const int64_t blk = slot / p.block_size;
  if (blk >= p.num_blocks) {
    if (tid == 0) set_device_error(p.err, 4u);
    return;
  }
  insert_latent<F>(p.cache + blk * p.block_stride + (slot % p.block_size) * p.entry_stride, p.kv_c + t * p.kv_s0, kr,
                   cs, (F == 1) ? *p.cache_scale_inv : 1.f, tid);
}

cudaError_t launch_prefill_epilogue(int fmt, const PrefillEpiParams& p, int Tp, cudaStream_t stream) {
  const dim3 grid(Tp, (p.H + 3) / 4);
  if (fmt == 0)
    mla_prefill_epilogue_kernel<0><<<grid, 128, 0, stream>>>(p);
  else if (fmt == 1)
    mla_prefill_epilogue_kernel<1><<<grid, 128, 0, stream>>>(p);
  else
    mla_prefill_epilogue_kernel<2><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Split-K merge: out = sum_s exp(lse_s - lse) * O_s, lse = ln sum_s exp(lse_s).  The same
// combine as vLLM's merge_attn_states ("vllm.models.kimi_k3.nvidia.mla",
// _forward_prefill_fused) applied across the key splits of one decode row, or of one sparse
// row (with an optional per-head sink logit e^{sink} added to the denominator).  One CTA of
// 128 threads per (row, head); each thread owns 4 of the 512 columns and keeps kBatch splits'
// loads in flight (the launch picks the smallest batch that covers the split count, since a
// larger one costs registers and so resident CTAs).
template <int kBatch>
__global__ void __launch_bounds__(128) mla_merge_kernel(const MergeParams p) {
  // launched as a programmatic dependent of the attention kernel: wait until its grid has
  // finished and its partials are visible (a no-op under an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t rh = blockIdx.x;
  const int64_t stride = static_cast<int64_t>(p.n_rows) * p.H;
  const int row = static_cast<int>(rh / p.H), h = static_cast<int>(rh % p.H);
  int S = p.S;
  if (p.seq_lens) {     // splits past the request's length hold nothing
    const int64_t L = max(p.seq_lens[row / p.q_len], 0);
    S = static_cast<int>(min(static_cast<int64_t>(S), (L + p.chunk - 1) / p.chunk));
  }
  // the split weights exp(lse_s - max) are formed once: thread s loads the LSE of split s
  // (and of s + 128, ...) once
  __shared__ float wsh[128];
  __shared__ float red[2][4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t lbase = rh;
  const float ls0 = tid < S ? p.part_lse[tid * stride + lbase] : -CUDART_INF_F;
  float m = ls0;
  for (int s = tid + 128; s < S; s += 128) m = fmaxf(m, p.part_lse[s * stride + lbase]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) red[0][warp] = m;
  __syncthreads();
  m = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
  // a sink logit joins the denominator with a zero value
  const float sk = p.sink ? p.sink[h] : -CUDART_INF_F;
  m = fmaxf(m, sk);
  auto weight = [&](float ls) { return (m == -CUDART_INF_F || ls == -CUDART_INF_F) ? 0.f : expf(ls - m); };
  const float w0 = weight(ls0);
  wsh[tid] = w0;
  float ws = w0 + ((tid == 0 && sk != -CUDART_INF_F) ? expf(sk - m) : 0.f);
  for (int s = tid + 128; s < S; s += 128) ws += weight(p.part_lse[s * stride + lbase]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ws += __shfl_xor_sync(0xFFFFFFFFu, ws, o);
  if (lane == 0) red[1][warp] = ws;
  __syncthreads();
  const float wsum = (red[1][0] + red[1][1]) + (red[1][2] + red[1][3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* po = reinterpret_cast<const float4*>(p.part_o + rh * 512) + tid;
  const int64_t step4 = stride * 128;      // one split, in float4
  for (int s0 = 0; s0 < S; s0 += kBatch) {
    float wb[kBatch];
    float4 ob[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int ss = s0 + u;
      wb[u] = ss >= S ? 0.f : ss < 128 ? wsh[ss] : weight(p.part_lse[ss * stride + lbase]);
      ob[u] = wb[u] != 0.f ? po[ss * step4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      acc.x += wb[u] * ob[u].x;
      acc.y += wb[u] * ob[u].y;
      acc.z += wb[u] * ob[u].z;
      acc.w += wb[u] * ob[u].w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out + row * p.o_s0b + h * p.o_s1b) + 4 * tid;
  dst[0] = __float2bfloat16_rn(acc.x * inv);
  dst[1] = __float2bfloat16_rn(acc.y * inv);
  dst[2] = __float2bfloat16_rn(acc.z * inv);
  dst[3] = __float2bfloat16_rn(acc.w * inv);
  if (tid == 0 && p.lse) p.lse[rh] = wsum > 0.f ? m + logf(wsum) : -CUDART_INF_F;
}

// ------------------------------------------------------------------------------------------
// Gather and dequantise: one warp per slot, 18 values per lane.
template <int F>
__global__ void mla_gather_kernel(const GatherParams p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (i >= p.n) return;
  const int lane = threadIdx.x & 31;
  const int64_t slot = p.slots[i];
  const uint8_t* ent = nullptr;
  if (slot >= 0) {
    const int64_t blk = slot / p.block_size;
    if (blk < p.num_blocks)
      ent = p.cache + blk * p.block_stride + (slot % p.block_size) * p.entry_stride;
    else if (lane == 0)
      set_device_error(p.err, 2u);
  }
  float* o = p.out + i * 576;
  for (int d = lane; d < 576; d += 32) {
    float v = 0.f;
    if (ent) {
      if (F == 0) {
        v = bf16_at(reinterpret_cast<const uint16_t*>(ent) + d);
      } else if (F == 1) {
        __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(ent[d]), __NV_E4M3);
        v = __half2float(__half(h));
      } else if (d < 512) {
        __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(ent[d]), __NV_E4M3);
        v = __half2float(__half(h)) * reinterpret_cast<const float*>(ent + 512)[d >> 7];
      } else {
        v = bf16_at(reinterpret_cast<const uint16_t*>(ent + 528) + (d - 512));
      }
    }
    o[d] = v;
  }
}

// ------------------------------------------------------------------------------------------
cudaError_t launch_epilogue(int fmt, const EpiParams& p, int B, cudaStream_t stream) {
  const dim3 grid(B, (p.H + 3) / 4 + 1);
  if (fmt == 0)
    mla_epilogue_kernel<0><<<grid, 128, 0, stream>>>(p);
  else if (fmt == 1)
    mla_epilogue_kernel<1><<<grid, 128, 0, stream>>>(p);
  else
    mla_epilogue_kernel<2><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// Scheduler reset: zero the work-item counter of a persistent decode kernel.  Chained to the
// kernels on either side as programmatic dependents (it waits for the previous kernel, so the
// decode kernel's own wait covers both), it lets the decode's setup overlap the epilogue.
__global__ void mla_sched_reset_kernel(uint32_t* sched) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) *sched = 0u;
}

cudaError_t launch_sched_reset(uint32_t* sched, cudaStream_t stream) {
  return launch_pdl(mla_sched_reset_kernel, dim3(1), dim3(32), 0, stream, sched);
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(p.n_rows) * p.H;
  if (n == 0) return cudaSuccess;
  // programmatic dependent launch: the merge CTAs are scheduled while the attention kernel's
  // last CTAs finish, and wait on the device instead of behind a launch gap
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(n));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.S <= 4) return cudaLaunchKernelEx(&cfg, mla_merge_kernel<4>, p);
  if (p.S <= 8) return cudaLaunchKernelEx(&cfg, mla_merge_kernel<8>, p);
  return cudaLaunchKernelEx(&cfg, mla_merge_kernel<16>, p);
}

cudaError_t launch_gather(int fmt, const GatherParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((p.n + 3) / 4);
  if (fmt == 0)
    mla_gather_kernel<0><<<grid, 128, 0, stream>>>(p);
  else if (fmt == 1)
    mla_gather_kernel<1><<<grid, 128, 0, stream>>>(p);
  else
    mla_gather_kernel<2><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Chunked-context gather.  "vllm.models.kimi_k3.nvidia.mla", _gather_context_latent: request b
// of a chunk owns rows cu[b] .. cu[b+1]-1; row cu[b] + i is context position starts[b] + i of
// request b, found through its block-table row.  kind 0 writes the 576 values as bf16 (fp8
// codes times their scale in fp32, rounded once; bf16 entries as stored), kind 1 the stored
// entry bytes.  One warp per row, 16-byte pieces per lane.

__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 c, float scale, uint4 (&o)[2]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> (16 * hh)), __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));     // exact
      r[2 * i + hh] = static_cast<uint32_t>(bf16_bits(f.x * scale)) | (static_cast<uint32_t>(bf16_bits(f.y * scale)) << 16);
    }
  }
  o[0] = make_uint4(r[0], r[1], r[2], r[3]);
  o[1] = make_uint4(r[4], r[5], r[6], r[7]);
}

template <int F, int KIND>
__global__ void __launch_bounds__(128) mla_gather_context_kernel(const GatherCtxParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (r >= p.num_tokens || r >= p.cu[p.batch]) return;
  int lo = 0, hi = p.batch - 1;           // the last request b with cu[b] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu[mid] <= r) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int64_t pos = (p.starts ? p.starts[b] : 0) + (r - p.cu[b]);
  const int64_t blk = p.block_table[static_cast<int64_t>(b) * p.bt_stride + pos / p.block_size];
  constexpr int kEntry = F == 0 ? 1152 : F == 1 ? 576 : 656;
  constexpr int kOut = KIND == 1 ? kEntry : 1152;
  uint8_t* dst = p.dst + r * p.dst_row;
  if (blk < 0 || blk >= p.num_blocks) {
    if (lane == 0) set_device_error(p.err, 2u);
    for (int i = lane; i < kOut; i += 32) dst[i] = 0;
    return;
  }
  const uint8_t* ent = p.cache + blk * p.block_stride + (pos % p.block_size) * p.entry_stride;
  if (!p.vec) {
    if (KIND == 1 || F == 0) {
      for (int i = lane; i < kEntry; i += 32) dst[i] = ent[i];
    } else {
      uint16_t* o = reinterpret_cast<uint16_t*>(dst);
      for (int d = lane; d < 576; d += 32) {
        float x;
        if (F == 1) {
          x = __half2float(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(ent[d]), __NV_E4M3)) * p.scale;
          o[d] = bf16_bits(x);
        } else if (d < 512) {
          const float sj = *reinterpret_cast<const float*>(ent + 512 + 4 * (d >> 7));
          o[d] = bf16_bits(__half2float(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(ent[d]), __NV_E4M3)) * sj);
        } else {
          o[d] = static_cast<uint16_t>(ent[528 + 2 * (d - 512)] | (ent[529 + 2 * (d - 512)] << 8));
        }
      }
    }
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(ent);
  uint4* out = reinterpret_cast<uint4*>(dst);
  if (KIND == 1 || F == 0) {
    for (int i = lane; i < kEntry / 16; i += 32) out[i] = __ldg(src + i);
  } else if (F == 1) {
    for (int i = lane; i < 36; i += 32) {       // 16 codes -> 16 bf16 values
      uint4 o[2];
      e4m3x16_to_bf16(__ldg(src + i), p.scale, o);
      out[2 * i] = o[0];
      out[2 * i + 1] = o[1];
    }
  } else {
    uint4 o[2];
    const float sj = __ldg(reinterpret_cast<const float*>(ent + 512) + (lane >> 3));
    e4m3x16_to_bf16(__ldg(src + lane), sj, o);
    out[2 * lane] = o[0];
    out[2 * lane + 1] = o[1];
    if (lane < 8) out[64 + lane] = __ldg(src + 33 + lane);     // rope bytes 528.. -> values 512..
  }
}

cudaError_t launch_gather_context(int fmt, int kind, const GatherCtxParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((p.num_tokens + 3) / 4);
  if (kind == 1) {
    if (fmt == 0) mla_gather_context_kernel<0, 1><<<grid, 128, 0, stream>>>(p);
    else if (fmt == 1) mla_gather_context_kernel<1, 1><<<grid, 128, 0, stream>>>(p);
    else mla_gather_context_kernel<2, 1><<<grid, 128, 0, stream>>>(p);
  } else {
    if (fmt == 0) mla_gather_context_kernel<0, 0><<<grid, 128, 0, stream>>>(p);
    else if (fmt == 1) mla_gather_context_kernel<1, 0><<<grid, 128, 0, stream>>>(p);
    else mla_gather_context_kernel<2, 0><<<grid, 128, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// merge_attn_states ("vllm.models.kimi_k3.nvidia.mla", _forward_prefill_fused): the context
// (prefix) and new-token (suffix) partials of prefill attention combined by their LSEs,
//   lse = ln(e^{lse_p} + e^{lse_s}),  out = e^{lse_p - lse} O_p + e^{lse_s - lse} O_s,
// in fp32, rounded once to bf16; both empty (-inf) -> 0 and -inf.  One warp per (token,
// head), 8 values per lane per step.
__global__ void __launch_bounds__(128) mla_merge_states_kernel(const MergeStatesParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t th = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (th >= static_cast<int64_t>(p.T) * p.H) return;
  const int t = static_cast<int>(th / p.H), h = static_cast<int>(th % p.H);
  const float lp = p.prefix_lse[static_cast<int64_t>(h) * p.T + t];
  const float ls = p.suffix_lse[static_cast<int64_t>(h) * p.T + t];
  const float m = fmaxf(lp, ls);
  float wp = 0.f, ws = 0.f, lse = -CUDART_INF_F;
  if (m != -CUDART_INF_F) {
    const float ep = expf(lp - m), es = expf(ls - m);
    const float inv = 1.f / (ep + es);
    wp = ep * inv;
    ws = es * inv;
    lse = m + logf(ep + es);
  }
  const uint16_t* a = p.prefix + t * p.p_s0 + h * p.p_s1;
  const uint16_t* c = p.suffix + t * p.s_s0 + h * p.s_s1;
  uint16_t* o = p.out + t * p.o_s0 + h * p.o_s1;
  if (p.vec) {
    for (int d0 = 8 * lane; d0 < p.D; d0 += 256) {
      const uint4 va = __ldg(reinterpret_cast<const uint4*>(a + d0));
      const uint4 vc = __ldg(reinterpret_cast<const uint4*>(c + d0));
      const uint32_t xa[4] = {va.x, va.y, va.z, va.w}, xc[4] = {vc.x, vc.y, vc.z, vc.w};
      uint32_t r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = wp * __uint_as_float(xa[i] << 16) + ws * __uint_as_float(xc[i] << 16);
        const float hi = wp * __uint_as_float(xa[i] & 0xFFFF0000u) + ws * __uint_as_float(xc[i] & 0xFFFF0000u);
        r[i] = static_cast<uint32_t>(bf16_bits(lo)) | (static_cast<uint32_t>(bf16_bits(hi)) << 16);
      }
      *reinterpret_cast<uint4*>(o + d0) = make_uint4(r[0], r[1], r[2], r[3]);
    }
  } else {
    for (int d = lane; d < p.D; d += 32) o[d] = bf16_bits(wp * bf16_at(a + d) + ws * bf16_at(c + d));
  }
  if (lane == 0 && p.out_lse) p.out_lse[static_cast<int64_t>(h) * p.T + t] = lse;
}

cudaError_t launch_merge_states(const MergeStatesParams& p, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(p.T) * p.H;
  mla_merge_states_kernel<<<static_cast<unsigned>((n + 3) / 4), 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
