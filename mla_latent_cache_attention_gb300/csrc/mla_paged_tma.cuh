// mla_paged_tma.cuh -- paged MLA decode / spec-verify over bf16 and plain-fp8 caches.
//
// What it computes ("FlashMLA: Multi-head Latent Attention decode kernels", decode with an
// absorbed query over the 576-wide latent cache; "vLLM MLA backend", paged decode with
// spec-verify query tokens): for every request b and query token qi, attention of the
// absorbed query q[b, qi, h, 0:576] over the keys at positions 0 .. L_b - q_len + qi of the
// paged cache (each key is the 576-wide latent [kv_c_normed | k_pe], the value its first 512),
// softmax scale applied to the logits, output O / l in bf16 and the natural-log LSE.
//
// How (GB300 design):
//   * One work item = one request x one group of NQ query columns (a column is one
//     (query token, head) pair) x one split of the key range.  Taking all q_len x H columns of
//     a request in one item reads the request's keys once for every query token and head.
//   * Key tiles of 128 keys are loaded by the tensor memory accelerator straight from the
//     pages: a 3-D tensor map [num_blocks][block_size][entry bytes] with 128-byte swizzle and
//     boxes of 128 bytes x BR rows, so every box lands in the canonical operand layout of a
//     128-row block and no thread touches the data on its way to the tensor core.  Pages past
//     the item's end or with an out-of-range id are loaded from an out-of-range block
//     coordinate, which fills zeros.  Blocks stream through a ring of 16 KB slots with
//     per-slot full / empty barriers, so loads run ahead of the MMAs across tiles and items.
//   * Products on the 5th-generation tensor cores with the key tile as the M = 128 operand
//     and the query columns as N (swap-AB): S^T = K Q^T and O^T += V^T P, accumulators in
//     TMEM.  bf16: kind::f16.  fp8: kind::f8f6f4 directly on the cache's e4m3 bytes (exact
//     products, fp32 accumulation); P is passed as two e4m3 terms hi + lo of 256 p, which
//     carries p to about 2^-8 relative, and both terms accumulate into the same O.
//   * fp8 issues QK of tile t+1 before PV of tile t (double-buffered S), so the softmax of a
//     tile overlaps the tensor pipe.  bf16 tiles are 144 KB, two do not fit, and the MMAs run
//     QK(t), PV(t) while the ring refills.
//   * Work items come from an atomic counter (longest splits first) when a scheduler word is
//     given, else by static striding.
//
// Warps: 0 producer (TMA issue; lanes resolve page ids), 1 MMA issuer and TMEM owner, 2..
// softmax + epilogue (4 warps, or 8 when NQ = 64: two column halves per TMEM lane quadrant).
#pragma once
#include <cuda.h>

#include "mla_attn.cuh"

namespace mla {

struct PagedParams {
  int H, q_len, B, G;           // G column groups of NQ columns per request
  int cols;                     // H * q_len
  int qbox_h, qbox_q;           // query TMA box: heads x tokens (rows = qbox_h * qbox_q <= NQ)
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;
  int num_blocks, block_size, BR;
  int chunk, n_splits, n_items;
  int n_rows;                   // B * q_len
  float sig2, out_scale;
  uint8_t* out;                 // bf16 [n_rows, H, >=512]
  int64_t o_s0b, o_s1b;
  float* lse;                   // [n_rows, H] or null
  float* part_o;                // [n_splits][n_rows][H][512] fp32 (n_splits > 1)
  float* part_lse;              // [n_splits][n_rows][H]
  uint32_t* sched;              // item counter, zero at launch; null: static striding
  uint32_t* err;
};

struct WorkItem {
  int b, g, s, ntiles, k0, n, L, pad;
};

constexpr int kItemDepth = 4;
constexpr int kSlotBytes = kTile * 128;

template <int F, int NQ>
struct PagedCfg {
  static_assert(F == kBF16 || F == kFP8, "format");
  static_assert(NQ == 16 || NQ == 32 || NQ == 64, "columns per item");
  static constexpr int kNB = F == kBF16 ? 10 : 5;        // ring positions per tile (bf16: 9 blocks + 1 pad)
  static constexpr int kNBQ = F == kBF16 ? 9 : 5;        // query blocks
  static constexpr int kRope = F == kBF16 ? 8 : 4;       // block used by QK only
  static constexpr int kSW = NQ == 64 ? 8 : 4;           // softmax warps
  static constexpr int kNC = NQ * 4 / kSW;               // columns per softmax thread
  static constexpr int kThreads = 64 + 32 * kSW;
  static constexpr bool kOverlap = F == kFP8;
  static constexpr int kQBytes = kNBQ * NQ * 128;
  static constexpr int kPBytes = F == kBF16 ? kTile * NQ * 2 : 2 * kTile * NQ;
  static constexpr int kRedBytes = 3 * NQ * 4 * 4;       // max partials [2][NQ][4], sum partials [NQ][4]
  static constexpr int kFixed = kQBytes + kPBytes + kRedBytes + kItemDepth * 32 + 8 * (9 + 2 * kItemDepth) + 64;
  static constexpr int ring_slots() {
    int r = (kSmemLimit - 1024 - kFixed) / (kSlotBytes + 16);
    if (F == kBF16 && (r & 1)) --r;                      // V pairs never wrap the ring
    return r;
  }
  static constexpr int kR = ring_slots();
  static_assert(kR >= 2 * kNB || (!kOverlap && kR >= kNB), "ring too small");
  static_assert(!kOverlap || kR >= 2 * kNB, "overlap needs two tiles in the ring");
  static constexpr int kRing = 0;
  static constexpr int kQ = kRing + kR * kSlotBytes;
  static constexpr int kP = kQ + kQBytes;
  static constexpr int kRed = kP + kPBytes;
  static constexpr int kItems = kRed + kRedBytes;
  static constexpr int kBar = kItems + kItemDepth * 32;
  static constexpr int kNumBars = 2 * kR + 9 + 2 * kItemDepth;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= kSmemLimit, "shared memory budget");
  static constexpr int kTmemS = 0, kTmemO = 2 * NQ;
  static constexpr int kTmemCols = 6 * NQ <= 128 ? 128 : 6 * NQ <= 256 ? 256 : 512;
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// D(tmem) (+)= A x B with e4m3 operands (kind::f8f6f4), fp32 accumulate.
__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4 with e4m3 A and B (format code 0), fp32 D.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

template <int NC>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float (&v)[NC]) {
#pragma unroll
  for (int u = 0; u < NC / 16; ++u) {
    float t[16];
    tmem_ld16(taddr + 16 * u, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[16 * u + i] = t[i];
  }
}
template <int NC>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const float (&v)[NC]) {
#pragma unroll
  for (int u = 0; u < NC / 16; ++u) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = v[16 * u + i];
    tmem_st16(taddr + 16 * u, t);
  }
}

// Transposing butterfly over the warp: on entry lane l holds NC values (one per column) of
// its own key; on exit lane l holds the reduction over all 32 lanes of column (l % NC).
template <int NC, bool kMax>
__device__ __forceinline__ float warp_col_reduce(float (&v)[NC], int lane) {
#pragma unroll
  for (int w = NC / 2; w >= 1; w /= 2) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float a = v[i], b = v[i + w];
      const float send = upper ? a : b;
      const float keep = upper ? b : a;
      const float r = __shfl_xor_sync(0xFFFFFFFFu, send, w);
      v[i] = kMax ? fmaxf(keep, r) : keep + r;
    }
  }
  float x = v[0];
  if (NC == 16) {
    const float r = __shfl_xor_sync(0xFFFFFFFFu, x, 16);
    x = kMax ? fmaxf(x, r) : x + r;
  }
  return x;
}

__device__ __forceinline__ uint32_t e4m3x2_sat(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

template <int F, int NQ>
__global__ void __launch_bounds__(PagedCfg<F, NQ>::kThreads, 1)
    mla_paged_tma_kernel(const __grid_constant__ PagedParams p, const __grid_constant__ CUtensorMap tm_kv,
                         const __grid_constant__ CUtensorMap tm_q) {
  using C = PagedCfg<F, NQ>;
  constexpr int R = C::kR, NB = C::kNB, NC = C::kNC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + C::kRing;
  uint8_t* qs = smem + C::kQ;
  uint8_t* ps = smem + C::kP;
  float* red = reinterpret_cast<float*>(smem + C::kRed);
  WorkItem* items = reinterpret_cast<WorkItem*>(smem + C::kItems);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + R;
  uint64_t* s_full = bars + 2 * R;        // [2]
  uint64_t* p_full = bars + 2 * R + 2;
  uint64_t* pv_done = bars + 2 * R + 3;
  uint64_t* q_full = bars + 2 * R + 4;
  uint64_t* q_empty = bars + 2 * R + 5;
  uint64_t* fin = bars + 2 * R + 6;
  uint64_t* item_full = bars + 2 * R + 9;
  uint64_t* item_empty = item_full + kItemDepth;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  TL_DECL;

  // query rows that no box writes stay zero
  for (int i = tid; i < C::kQBytes / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(qs)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 1);
    mbar_init(pv_done, 1);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(fin, 1);
    for (int k = 0; k < kItemDepth; ++k) {
      mbar_init(&item_full[k], 1);
      mbar_init(&item_empty[k], 2);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const int NPG = kTile / p.BR;
    uint32_t errbits = 0;
    int64_t pos = 0;   // ring positions issued
    int nitem = 0, nq = 0;
    bool ok = true;
    int ticket = 0;
    if (lane == 0) ticket = p.sched ? static_cast<int>(atomicAdd(p.sched, 1u)) : static_cast<int>(blockIdx.x);
    ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
    int stride_k = 1;
    while (ok) {
      const int item = ticket;
      if (item >= p.n_items) break;
      if (lane == 0)
        ticket = p.sched ? static_cast<int>(atomicAdd(p.sched, 1u)) : static_cast<int>(blockIdx.x + stride_k * gridDim.x);
      ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
      ++stride_k;
      WorkItem it;
      const int bg = p.B * p.G;
      it.s = item / bg;
      it.b = (item % bg) / p.G;
      it.g = item % p.G;
      it.L = max(p.seq_lens[it.b], 0);
      it.k0 = it.s * p.chunk;
      it.n = min(max(it.L - it.k0, 0), p.chunk);
      it.ntiles = (it.n + kTile - 1) / kTile;
      it.pad = 0;
      if (it.n == 0 && p.n_splits > 1) continue;     // an empty split: the merge skips it
      {
        const int k = nitem % kItemDepth;
        if (nitem >= kItemDepth && !mbar_wait(&item_empty[k], ((nitem / kItemDepth) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          items[k] = it;
          mbar_arrive(&item_full[k]);
        }
        ++nitem;
      }
      if (it.ntiles == 0) continue;
      // query columns of the item: box (128 B x qbox_h heads x qbox_q tokens) per block
      if (nq > 0 && !mbar_wait(q_empty, (nq - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const int cg0 = it.g * NQ;
        const int h0 = cg0 % p.H, r0 = it.b * p.q_len + cg0 / p.H;
        mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(C::kNBQ * 128 * p.qbox_h * p.qbox_q));
#pragma unroll 1
        for (int blk = 0; blk < C::kNBQ; ++blk) {
          const int x = (F == kFP8 && blk == 4) ? 448 : 128 * blk;
          tma_load_3d(qs + blk * NQ * 128, &tm_q, x, h0, r0, q_full);
        }
      }
      ++nq;
      for (int t = 0; t < it.ntiles && ok; ++t) {
        // page ids of the tile (lane q < NPG holds page q); out-of-range -> zero-filled box
        int blk = p.num_blocks, y = 0;
        if (lane < NPG) {
          const int kp = it.k0 + t * kTile + lane * p.BR;
          if (kp < it.k0 + it.n) {
            const int id = p.block_table[static_cast<int64_t>(it.b) * p.bt_stride + kp / p.block_size];
            if (id >= 0 && id < p.num_blocks) {
              blk = id;
              y = kp % p.block_size;
            } else {
              errbits |= 2u;
            }
          }
        }
        if (lane == 0) TL(0, 1);
#pragma unroll 1
        for (int b = 0; b < NB; ++b, ++pos) {
          const int slot = static_cast<int>(pos % R);
          const int use = static_cast<int>(pos / R);
          if (use > 0 && !mbar_wait(&empty[slot], (use - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          if (F == kBF16 && b == 9) {
            if (lane == 0) mbar_arrive(&full[slot]);
            continue;
          }
          if (lane == 0) mbar_arrive_expect_tx(&full[slot], kSlotBytes);
          __syncwarp();
          const int x = (F == kFP8 && b == 4) ? 448 : 128 * b;
          for (int q = 0; q < NPG; ++q) {
            const int z = __shfl_sync(0xFFFFFFFFu, blk, q);
            const int yy = __shfl_sync(0xFFFFFFFFu, y, q);
            if (lane == 0) tma_load_3d(ring + slot * kSlotBytes + q * p.BR * 128, &tm_kv, x, yy, z, &full[slot]);
          }
        }
      }
    }
    // end marker
    if (ok) {
      const int k = nitem % kItemDepth;
      if (nitem < kItemDepth || mbar_wait(&item_empty[k], ((nitem / kItemDepth) - 1) & 1, abort_flag)) {
        if (lane == 0) {
          WorkItem e{};
          e.b = -1;
          items[k] = e;
          mbar_arrive(&item_full[k]);
        }
      }
    }
    // never leave copies in flight behind us
    {
      volatile int no_abort = 0;
      const int64_t first = pos > R ? pos - R : 0;
      for (int64_t q = first; q < pos; ++q) {
        const int slot = static_cast<int>(q % R);
        mbar_wait(&full[slot], static_cast<uint32_t>(q / R) & 1u, &no_abort);
      }
      if (nq > 0) mbar_wait(q_full, (nq - 1) & 1, &no_abort);
    }
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (lane == 0 && errbits) set_device_error(p.err, errbits);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t ring_a = smem_u32(ring), q_a = smem_u32(qs), p_a = smem_u32(ps);
      const uint64_t dK0 = smem_desc(ring_a, 16, 1024, kSwizzle128B);
      const uint64_t dQ0 = smem_desc(q_a, 16, 1024, kSwizzle128B);
      const uint64_t dV0 = smem_desc(ring_a, kSlotBytes, 1024, kSwizzle128B);
      constexpr uint32_t kPLbo = F == kBF16 ? NQ * 16 : NQ * 8;   // 8-key groups of P
      const uint64_t dP0 = smem_desc(p_a, kPLbo, 128, kSwizzleNone);
      constexpr uint32_t kIdQk = F == kBF16 ? idesc_f16(128, NQ, 1, 1, 0, 0) : idesc_e4m3(128, NQ, 0, 0);
      constexpr uint32_t kIdPv = F == kBF16 ? idesc_f16(128, NQ, 1, 1, 1, 1) : idesc_e4m3(128, NQ, 1, 1);
      auto slot_of = [&](int gt, int b) -> int { return static_cast<int>((static_cast<int64_t>(gt) * NB + b) % R); };
      auto use_of = [&](int gt, int b) -> uint32_t {
        return static_cast<uint32_t>(((static_cast<int64_t>(gt) * NB + b) / R) & 1);
      };
      bool ok = true;
      int nit = 0, nq = 0, g = 0;
      // QK of global tile gt into S buffer gt & 1; returns false on a failed wait
      auto issue_qk = [&](int gt, bool last) -> bool {
        const uint32_t dS = tmem + C::kTmemS + (gt & 1) * NQ;
        TL(2, 1);
#pragma unroll 1
        for (int b = 0; b < NB; ++b) {
          const int slot = slot_of(gt, b);
          if (!mbar_wait(&full[slot], use_of(gt, b), abort_flag)) return false;
          tc_fence_after();
          if (F == kBF16 && b == 9) {
            mbar_arrive(&empty[slot]);
            continue;
          }
          const uint64_t aK = dK0 + ((slot * kSlotBytes) >> 4);
          const uint64_t bQ = dQ0 + ((b * NQ * 128) >> 4);
          if (F == kBF16) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(dS, aK + ((kk * 32) >> 4), bQ + ((kk * 32) >> 4), kIdQk, (b > 0 || kk > 0) ? 1u : 0u);
          } else {
            const int kk0 = (b == 4) ? 2 : 0;      // block 4 holds elements 448..575; 512.. are new
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (kk >= kk0)
                mma_f8_ss(dS, aK + ((kk * 32) >> 4), bQ + ((kk * 32) >> 4), kIdQk, (b > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&s_full[gt & 1]);
        mma_commit(&empty[slot_of(gt, C::kRope)]);
        if (last) mma_commit(q_empty);
        TL(2, 2);
        return true;
      };
      auto issue_pv = [&](int gt, bool first) -> bool {
        if (!mbar_wait(p_full, static_cast<uint32_t>(gt) & 1u, abort_flag)) return false;
        tc_fence_after();
        TL(2, 3);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t dO = tmem + C::kTmemO + j * NQ;
          if (F == kBF16) {
            const uint64_t aV = dV0 + ((slot_of(gt, 2 * j) * kSlotBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ss(dO, aV + ((kk * 2048) >> 4), dP0 + ((kk * NQ * 32) >> 4), kIdPv, (!first || kk > 0) ? 1u : 0u);
            mma_commit(&empty[slot_of(gt, 2 * j)]);
            mma_commit(&empty[slot_of(gt, 2 * j + 1)]);
          } else {
            const uint64_t aV = dV0 + ((slot_of(gt, j) * kSlotBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t pb = dP0 + ((kk * NQ * 32) >> 4);
              mma_f8_ss(dO, aV + ((kk * 4096) >> 4), pb, kIdPv, (!first || kk > 0) ? 1u : 0u);
              mma_f8_ss(dO, aV + ((kk * 4096) >> 4), pb + ((kTile * NQ) >> 4), kIdPv, 1u);
            }
            mma_commit(&empty[slot_of(gt, j)]);
          }
        }
        mma_commit(pv_done);
        TL(2, 4);
        return true;
      };
      while (ok) {
        const int k = nit % kItemDepth;
        if (!mbar_wait(&item_full[k], (nit / kItemDepth) & 1, abort_flag)) break;
        const WorkItem it = items[k];
        mbar_arrive(&item_empty[k]);
        ++nit;
        if (it.b < 0) break;
        if (it.ntiles == 0) continue;
        if (!mbar_wait(q_full, nq & 1, abort_flag)) break;
        ++nq;
        tc_fence_after();
        if (C::kOverlap) {
          ok = issue_qk(g, it.ntiles == 1);
          for (int t = 1; t < it.ntiles && ok; ++t) {
            ok = issue_qk(g + t, t == it.ntiles - 1);
            ok = ok && issue_pv(g + t - 1, t == 1);
          }
          ok = ok && issue_pv(g + it.ntiles - 1, it.ntiles == 1);
        } else {
          for (int t = 0; t < it.ntiles && ok; ++t) {
            ok = issue_qk(g + t, t == it.ntiles - 1);
            ok = ok && issue_pv(g + t, t == 0);
          }
        }
        g += it.ntiles;
      }
      mma_commit(fin);
      volatile int no_abort = 0;
      mbar_wait(fin, 0, &no_abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    constexpr int NT = 32 * C::kSW;
    const int sw = warp - 2;
    const int quad = warp & 3;                  // TMEM lane quadrant of this warp
    const int c0 = (sw >> 2) * NC;              // first column of this thread
    const int row = quad * 32 + lane;           // key row of the tile / TMEM lane
    const int stid = tid - 64;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* red_m = red;                         // [2][NQ][4]
    float* red_l = red + 2 * NQ * 4;            // [NQ][4]
    constexpr float kPScale = F == kFP8 ? 8.f : 0.f;   // fp8: p carried as 256 p (log2 256 = 8)
    int nit = 0, g = 0;
    bool ok = true;
    while (ok) {
      const int k = nit % kItemDepth;
      bool w = mbar_wait(&item_full[k], (nit / kItemDepth) & 1, abort_flag);
      const WorkItem it = items[k];
      ++nit;
      if (!named_bar_and(1, NT, w)) break;
      if (it.b < 0) break;
      float m_run[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) m_run[c] = -CUDART_INF_F;
      float l_lane = 0.f;                         // this warp's keys' sum of p, column (lane % NC)
      const int cgb = it.g * NQ + c0;           // global column of this thread's column 0
      for (int t = 0; t < it.ntiles; ++t) {
        const int gt = g + t;
        w = mbar_wait(&s_full[gt & 1], static_cast<uint32_t>(gt >> 1) & 1u, abort_flag);
        tc_fence_after();
        if (stid == 0) TL(3, 1);
        float s[NC];
        tmem_ld_n<NC>(tl + C::kTmemS + (gt & 1) * NQ + c0, s);
        tmem_ld_wait();
        const int kpos = it.k0 + t * kTile + row;
        const bool rv = kpos < it.k0 + it.n;
#pragma unroll
        for (int c = 0; c < NC; ++c) s[c] = rv ? s[c] * p.sig2 : -CUDART_INF_F;
        // spec-verify: query token qi sees keys up to L - q_len + qi
        const int dq = kpos - it.L + p.q_len;
        if (rv && dq > 0) {
#pragma unroll
          for (int c = 0; c < NC; ++c)
            if ((cgb + c) / p.H < dq) s[c] = -CUDART_INF_F;
        }
        // rows past the item never reach PV with stale contents
        if (!rv && c0 == 0) {
#pragma unroll 1
          for (int b = 0; b < (F == kBF16 ? 8 : 4); ++b) {
            uint4* dst = reinterpret_cast<uint4*>(
                ring + static_cast<int>((static_cast<int64_t>(gt) * NB + b) % R) * kSlotBytes + row * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          }
        }
        float* rb = red_m + (gt & 1) * NQ * 4;
        {
          float v[NC];
#pragma unroll
          for (int c = 0; c < NC; ++c) v[c] = s[c];
          const float wm = warp_col_reduce<NC, true>(v, lane);
          if (NC == 32 || lane < 16) rb[(c0 + (lane % NC)) * 4 + quad] = wm;
        }
        ok = named_bar_and(1, NT, w);
        if (!ok) break;
        bool changed = false;
        float alpha[NC];
        float alpha_lane = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float4 q4 = reinterpret_cast<const float4*>(rb)[c0 + c];
          const float mt = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
          const float mnew = fmaxf(m_run[c], mt);
          const float mu = (mnew == -CUDART_INF_F) ? 0.f : mnew;
          alpha[c] = exp2f(m_run[c] - mu);
          s[c] = exp2f(s[c] - mu + kPScale);     // p (fp8: 256 p)
          if (c == (lane % NC)) alpha_lane = alpha[c];
          changed |= (mnew != m_run[c]);
          m_run[c] = mnew;
        }
        if (stid == 0) TL(3, 2);
        if (t > 0) {
          w = mbar_wait(pv_done, static_cast<uint32_t>(gt - 1) & 1u, abort_flag);   // PV of the previous tile
          tc_fence_after();
          if (w && changed) {
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
              float o[NC];
              tmem_ld_n<NC>(tl + C::kTmemO + j * NQ + c0, o);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < NC; ++c) o[c] *= alpha[c];
              tmem_st_n<NC>(tl + C::kTmemO + j * NQ + c0, o);
            }
            tmem_st_wait();
          }
        }
        if (F == kBF16) {
          // MN-major no-swizzle: 8 keys x 8 columns core matrices, 8-key groups NQ*16 bytes apart
#pragma unroll
          for (int c = 0; c < NC; c += 8) {
            uint4 v;
            v.x = pack2(s[c + 0], s[c + 1], true);
            v.y = pack2(s[c + 2], s[c + 3], true);
            v.z = pack2(s[c + 4], s[c + 5], true);
            v.w = pack2(s[c + 6], s[c + 7], true);
            *reinterpret_cast<uint4*>(ps + (row >> 3) * (NQ * 16) + (row & 7) * 16 + ((c0 + c) >> 3) * 128) = v;
          }
        } else {
          // 8 keys x 16 columns core matrices, 8-key groups NQ*8 bytes apart; hi then lo
#pragma unroll
          for (int c = 0; c < NC; c += 16) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float a0 = s[c + 4 * u], a1 = s[c + 4 * u + 1], a2 = s[c + 4 * u + 2], a3 = s[c + 4 * u + 3];
              const uint32_t h01 = e4m3x2_sat(a0, a1), h23 = e4m3x2_sat(a2, a3);
              const float2 f01 = e4m3x2_to_float2(h01), f23 = e4m3x2_to_float2(h23);
              const uint32_t l01 = e4m3x2_sat(a0 - f01.x, a1 - f01.y), l23 = e4m3x2_sat(a2 - f23.x, a3 - f23.y);
              hw[u] = h01 | (h23 << 16);
              lw[u] = l01 | (l23 << 16);
            }
            const int off = (row >> 3) * (NQ * 8) + (row & 7) * 16 + ((c0 + c) >> 4) * 128;
            *reinterpret_cast<uint4*>(ps + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(ps + kTile * NQ + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = named_bar_and(1, NT, w);
        if (!ok) break;
        if (stid == 0) mbar_arrive(p_full);
        if (stid == 0) TL(3, 3);
        // row sums of the tile while PV runs
        l_lane = l_lane * alpha_lane + warp_col_reduce<NC, false>(s, lane);
      }
      if (!ok) break;
      // ---- epilogue: O / l and the LSE of every column of the item
      w = true;
      if (it.ntiles > 0) {
        w = mbar_wait(pv_done, static_cast<uint32_t>(g + it.ntiles - 1) & 1u, abort_flag);
        tc_fence_after();
      }
      g += it.ntiles;
      if (NC == 32 || lane < 16) red_l[(c0 + (lane % NC)) * 4 + quad] = l_lane;
      ok = named_bar_and(1, NT, w);
      if (!ok) break;
      float inv[NC];
      float lse_mine = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const float4 q4 = reinterpret_cast<const float4*>(red_l)[c0 + c];
        const float l = (q4.x + q4.y) + (q4.z + q4.w);
        const bool live = l > 0.f;
        inv[c] = live ? p.out_scale / l : 0.f;
        const float lse = live ? (m_run[c] + log2f(l) - kPScale) * 0.69314718055994531f : -CUDART_INF_F;
        if (c == row) lse_mine = lse;
      }
      const bool final_out = (p.n_splits == 1);
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        float o[NC];
        if (it.ntiles > 0) {
          tmem_ld_n<NC>(tl + C::kTmemO + j * NQ + c0, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < NC; ++c) o[c] = 0.f;
        }
        const int d = 128 * j + row;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int cg = cgb + c;
          if (cg < p.cols) {
            const int orow = it.b * p.q_len + cg / p.H, h = cg % p.H;
            const float val = o[c] * inv[c];
            if (final_out) {
              *reinterpret_cast<__nv_bfloat16*>(p.out + orow * p.o_s0b + h * p.o_s1b + 2 * d) = __float2bfloat16_rn(val);
            } else {
              p.part_o[((static_cast<int64_t>(it.s) * p.n_rows + orow) * p.H + h) * kLora + d] = val;
            }
          }
        }
      }
      if (row < NC && cgb + row < p.cols) {
        const int cg = cgb + row;
        const int orow = it.b * p.q_len + cg / p.H, h = cg % p.H;
        if (final_out) {
          if (p.lse) p.lse[static_cast<int64_t>(orow) * p.H + h] = lse_mine;
        } else {
          p.part_lse[(static_cast<int64_t>(it.s) * p.n_rows + orow) * p.H + h] = lse_mine;
        }
      }
      tc_fence_before();
      named_bar_sync(1, NT);
      if (stid == 0) mbar_arrive(&item_empty[k]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag == 2) set_device_error(p.err, 16u);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace mla
