// mla_paged_tma.cuh -- paged MLA decode / spec-verify over bf16 and plain-fp8 caches.
//
// What it computes ("vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.prepared",
// PreparedMla.stock_core and trtllm_decode: decode of q query tokens per request over the
// paged latent cache, causal among them, split count bounded by max_context; bmm1_scale =
// softmax_scale * q_scale * k_scale and bmm2_scale = k_scale for the plain fp8 cache): for
// every request b and query token qi, attention of the
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

// Pipeline choices (measured on GB300; the defaults are the fastest found):
//   MLA_OVERLAP_FP8  fp8 issues QK(t+1) before PV(t)
//   MLA_LOOKAHEAD    tiles between a page-table lookup and the tile's loads
//   MLA_L2PF         also prefetch that tile into L2 when its pages are known: 1 by tensor
//                    boxes, 2 by one bulk prefetch per page (its rows are contiguous)
//   MLA_SLOT_COMMITS release each bf16 ring slot by its own commit (else by PV of its tile)
//   MLA_PV_WARP      PV issued by a warp of its own (else by the QK issuer)
#ifndef MLA_OVERLAP_FP8
#define MLA_OVERLAP_FP8 1
#endif
#ifndef MLA_LOOKAHEAD
#define MLA_LOOKAHEAD 1
#endif
#ifndef MLA_L2PF
#define MLA_L2PF 2
#endif
#ifndef MLA_SLOT_COMMITS
#define MLA_SLOT_COMMITS 1
#endif
#ifndef MLA_PV_WARP
#define MLA_PV_WARP 1
#endif

namespace mla {

struct PagedParams {
  const uint8_t* kv;            // the cache (for whole-page L2 prefetches)
  int64_t kv_blk_stride, kv_ent_stride;
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
  int wait_us;                  // in-kernel wait limit (0: the default, about 1 s)
  int stall;                    // test aid: the producer issues no loads (every wait runs out)
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
  static constexpr int KM = kTile;                        // keys per tile (QK MMA M)
  static constexpr int kSlot = KM * 128;                  // one ring slot: KM rows of 128 B
  static constexpr int kNB = F == kBF16 ? 10 : 5;        // ring positions per tile (bf16: 9 blocks + 1 pad)
  static constexpr int kNBQ = F == kBF16 ? 9 : 5;        // query blocks
  static constexpr int kRope = F == kBF16 ? 8 : 4;       // block used by QK only
  static constexpr int kSW = NQ == 64 ? 8 : 4;           // softmax warps
  static constexpr int kNC = NQ * 4 / kSW;               // columns per softmax thread
  static constexpr bool kPvSplit = MLA_PV_WARP;
  static constexpr int kPvWarp = kPvSplit ? 2 + kSW : -1;   // after the softmax warps
  static constexpr int kThreads = 64 + 32 * kSW + (kPvSplit ? 32 : 0);
  static constexpr bool kOverlap = F == kFP8 && MLA_OVERLAP_FP8;
  static constexpr int kPfDist = MLA_LOOKAHEAD;           // tiles between a page lookup and its use
  static constexpr bool kL2Pf = MLA_L2PF;
  // per-slot release commits pay for bf16 (a 147 KB tile fits 1.2 times: its slots refill as
  // soon as each is done); fp8 (two tiles in the ring) is faster with one release per tile,
  // since every commit drains the MMA pipe
  static constexpr bool kSlotCommits = MLA_SLOT_COMMITS && F == kBF16;
  static constexpr int kQBytes = kNBQ * NQ * 128;
  static constexpr int kPBytes = F == kBF16 ? KM * NQ * 2 : 2 * KM * NQ;
  static constexpr int kRedBytes = 3 * NQ * 4 * 4 + 2 * NQ * 4;   // max / sum partials, reference max, rescale
  static constexpr int kFixed = kQBytes + kPBytes + kRedBytes + kItemDepth * 32 + 8 * (9 + 2 * kItemDepth) + 64;
  static constexpr int ring_slots() {
    int r = (kSmemLimit - 1024 - kFixed) / (kSlot + 16);
    if (F == kBF16 && (r & 1)) --r;                      // V pairs never wrap the ring
    return r;
  }
  static constexpr int kR = ring_slots();
  static_assert(kR >= 2 * kNB || (!kOverlap && kR >= kNB), "ring too small");
  static_assert(!kOverlap || kR >= 2 * kNB, "overlap needs two tiles in the ring");
  static constexpr int kRing = 0;
  static constexpr int kQ = kRing + kR * kSlot;
  static constexpr int kP = kQ + kQBytes;
  static constexpr int kRed = kP + kPBytes;
  static constexpr int kItems = kRed + kRedBytes;
  static constexpr int kBar = kItems + kItemDepth * 32;
  static constexpr int kNumBars = 2 * kR + 10 + 2 * kItemDepth;
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

// The same box written at the same offset into every CTA of `mask` (cluster multicast); each
// destination's mbarrier at `bar`'s offset receives the box's bytes.
__device__ __forceinline__ void tma_load_3d_mc(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, "
      "{%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

// Contiguous global bytes into L2 (address and size multiples of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* tm, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tm), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Bounded wait by lane 0 of the warp only (fewer shared-memory polls); its outcome and the
// acquired view reach the other lanes through the warp barrier.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  bool w = true;
  if ((threadIdx.x & 31) == 0) w = mbar_wait(bar, parity, abort_flag);
  w = __shfl_sync(0xFFFFFFFFu, w ? 1 : 0, 0) != 0;
  __syncwarp();
  return w;
}

// The same with acquire at cluster scope (phases completed by another CTA's arrivals).
__device__ __forceinline__ bool warp_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  bool w = true;
  if ((threadIdx.x & 31) == 0) w = mbar_wait_cl(bar, parity, abort_flag);
  w = __shfl_sync(0xFFFFFFFFu, w ? 1 : 0, 0) != 0;
  __syncwarp();
  return w;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// PV of tile gt (its first ring position is gt * NB): O_j (+)= V_j^T P for the four value
// blocks j.  The slot index wraps by one subtraction and the descriptors advance by 32-bit
// adds: the issuing thread shares its sub-partition with busy warps, so it is kept to a few
// instructions per MMA.  bf16 takes V_j from the slot pair (2j, 2j + 1): an even ring length
// keeps a pair from wrapping.
template <class C, int F, int NQ>
__device__ __forceinline__ void paged_issue_pv(uint32_t tmem, uint64_t dV0, uint64_t dP0, uint64_t* empty, int gt,
                                               bool first) {
  constexpr int R = C::kR, NB = C::kNB, KM = C::KM;
  constexpr uint32_t kIdPv = F == kBF16 ? idesc_f16(128, NQ, 1, 1, 1, 1) : idesc_e4m3(128, NQ, 1, 1);
  const int s0 = static_cast<int>((static_cast<int64_t>(gt) * NB) % R);
  const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t dO = tmem + C::kTmemO + j * NQ;
    int sa = s0 + (F == kBF16 ? 2 * j : j);
    if (sa >= R) sa -= R;
    const uint64_t aV = desc_add(dV0, static_cast<uint32_t>(sa) * (C::kSlot >> 4));
    if (F == kBF16) {
#pragma unroll
      for (int kk = 0; kk < KM / 16; ++kk)
        mma_f16_ss(dO, desc_add(aV, (kk * 2048) >> 4), desc_add(dP0, (kk * NQ * 32) >> 4), kIdPv, kk > 0 ? 1u : acc0);
      if (C::kSlotCommits) {
        mma_commit(&empty[sa]);
        mma_commit(&empty[sa + 1]);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < KM / 32; ++kk) {
        const uint64_t pb = desc_add(dP0, (kk * NQ * 32) >> 4);
        mma_f8_ss(dO, desc_add(aV, (kk * 4096) >> 4), pb, kIdPv, kk > 0 ? 1u : acc0);
        mma_f8_ss(dO, desc_add(aV, (kk * 4096) >> 4), desc_add(pb, (KM * NQ) >> 4), kIdPv, 1u);
      }
      if (C::kSlotCommits) mma_commit(&empty[sa]);
    }
  }
}

template <int F, int NQ>
__global__ void __launch_bounds__(PagedCfg<F, NQ>::kThreads, 1)
    mla_paged_tma_kernel(const __grid_constant__ PagedParams p, const __grid_constant__ CUtensorMap tm_kv,
                         const __grid_constant__ CUtensorMap tm_q) {
  using C = PagedCfg<F, NQ>;
  constexpr int R = C::kR, NB = C::kNB, NC = C::kNC, KM = C::KM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + C::kRing;
  uint8_t* qs = smem + C::kQ;
  uint8_t* ps = smem + C::kP;
  float* red = reinterpret_cast<float*>(smem + C::kRed);
  WorkItem* items = reinterpret_cast<WorkItem*>(smem + C::kItems);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  // Every tcgen05.commit costs the tensor pipe a drain, so the MMA side commits twice per tile
  // only: s_full[t & 1] after QK(t) and pv_done[t & 1] after PV(t).  A ring slot is free once
  // PV of the tile that last used it is done, and the query tile once QK of the item's last
  // tile is.
  uint64_t* full = bars;                  // [R] TMA landed
  uint64_t* s_full = bars + R;            // [2]
  uint64_t* pv_done = bars + R + 2;       // [2]
  uint64_t* p_full = bars + R + 4;
  uint64_t* q_full = bars + R + 5;
  uint64_t* fin = bars + R + 6;
  uint64_t* item_full = bars + R + 8;
  uint64_t* item_empty = item_full + kItemDepth;
  uint64_t* empty = item_empty + kItemDepth;  // [R] slot consumed (per-slot release)
  uint64_t* fin_pv = bars + R + 7;
  uint64_t* s_free = empty + R;           // [2] the softmax has read S[t & 1] (PV warp split)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  TL_DECL;

  // the split-K merge may be scheduled now; it waits for this grid to complete
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // query rows that no box writes stay zero
  for (int i = tid; i < C::kQBytes / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(qs)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(p_full, C::kSW);     // one arrival per softmax warp
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    mbar_init(fin_pv, 1);
    mbar_init(&s_free[0], 1);
    mbar_init(&s_free[1], 1);
    for (int k = 0; k < kItemDepth; ++k) {
      mbar_init(&item_full[k], 1);
      mbar_init(&item_empty[k], C::kPvSplit ? 3 : 2);
    }
    *abort_flag = 0;
    abort_flag[1] = p.wait_us;
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
  // launched as a programmatic dependent of the previous kernel in the stream: the setup above
  // overlaps that kernel's tail, and its writes (a decode epilogue's query and cache entry, the
  // scheduler reset) are visible past this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const int NPG = KM / p.BR;
    uint32_t errbits = 0;
    int64_t pos = 0;   // ring positions issued
    int nitem = 0, nq = 0, stride_k = 0;
    int gq = -1;       // global index of the last tile of the previous item with tiles
    int gt_next = 0;   // global index of the next tile
    int t_waited = -1; // last tile whose PV the producer waited for
    bool ok = true;
    // work items: decode a queue ticket (empty splits skipped: the merge ignores them)
    auto take_ticket = [&]() -> int {
      int item = 0;
      if (lane == 0)
        item = p.sched ? static_cast<int>(atomicAdd(p.sched, 1u)) : static_cast<int>(blockIdx.x + stride_k * gridDim.x);
      ++stride_k;
      return __shfl_sync(0xFFFFFFFFu, item, 0);
    };
    auto decode = [&](int item, WorkItem& it) -> bool {     // false: empty split
      it.b = -1;
      if (item >= p.n_items) return true;
      const int bg = p.B * p.G;
      it.s = item / bg;
      it.b = (item % bg) / p.G;
      it.g = item % p.G;
      it.L = max(p.seq_lens[it.b], 0);
      it.k0 = it.s * p.chunk;
      it.n = min(max(it.L - it.k0, 0), p.chunk);
      it.ntiles = (it.n + KM - 1) / KM;
      it.pad = 0;
      return it.n > 0 || p.n_splits == 1;
    };
    auto next_item = [&](int ticket) -> WorkItem {
      WorkItem it{};
      while (!decode(ticket, it)) ticket = take_ticket();
      return it;
    };
    // block_table entry of page q of tile t of an item (-1: past the item), issued early and
    // checked late so that its latency hides behind the copies in flight
    auto page_raw = [&](const WorkItem& it, int t, int q) -> int {
      if (it.b < 0 || t >= it.ntiles) return -2;
      const int kp = it.k0 + t * KM + q * p.BR;
      if (kp >= it.k0 + it.n) return -1;
      return p.block_table[static_cast<int64_t>(it.b) * p.bt_stride + kp / p.block_size];
    };
    auto page_fix = [&](const WorkItem& it, int t, int q, int raw, int& y) -> int {
      y = 0;
      if (raw == -1 || raw == -2) return p.num_blocks;
      if (raw < 0 || raw >= p.num_blocks) {
        errbits |= 2u;
        return p.num_blocks;
      }
      y = (it.k0 + t * KM + q * p.BR) % p.block_size;
      return raw;
    };
    constexpr int D = C::kPfDist;
    // resolved pages of the next D tiles in processing order (lane q < NPG: page q)
    int fb[D], fy[D];
    bool fv[D];
#pragma unroll
    for (int i = 0; i < D; ++i) fv[i] = false, fb[i] = 0, fy[i] = 0;
    // the next item is claimed only when the current one is D tiles from its end, so that
    // the queue hands the tail out evenly
    WorkItem cur = next_item(take_ticket());
    WorkItem nxt{};
    bool have_nxt = false;
    if (p.stall) {
      // test aid: hand the first item to the consumers and issue none of its loads, so that
      // their waits run out under the launch's short wait limit; no copy is ever in flight
      if (cur.b >= 0) {
        if (lane == 0) {
          items[0] = cur;
          mbar_arrive(&item_full[0]);
        }
        nitem = 1;
      }
      ok = false;
    }
    while (ok && cur.b >= 0) {
      {
        const int k = nitem % kItemDepth;
        if (nitem >= kItemDepth && !warp_wait(&item_empty[k], ((nitem / kItemDepth) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          items[k] = cur;
          mbar_arrive(&item_full[k]);
        }
        ++nitem;
      }
      if (lane == 0) TL(0, 5);
      if (cur.ntiles > 0) {
        // query columns of the item: box (128 B x qbox_h heads x qbox_q tokens) per block
        if (gq >= 0 && !warp_wait(&s_full[gq & 1], static_cast<uint32_t>(gq >> 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const int cg0 = cur.g * NQ;
          const int h0 = cg0 % p.H, r0 = cur.b * p.q_len + cg0 / p.H;
          mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(C::kNBQ * 128 * p.qbox_h * p.qbox_q));
#pragma unroll 1
          for (int blk = 0; blk < C::kNBQ; ++blk) {
            const int x = (F == kFP8 && blk == 4) ? 448 : 128 * blk;
            tma_load_3d(qs + blk * NQ * 128, &tm_q, x, h0, r0, q_full);
          }
        }
        ++nq;
      }
      for (int t = 0; t < cur.ntiles && ok; ++t) {
        if (!have_nxt && t + D >= cur.ntiles) {
          nxt = next_item(take_ticket());
          have_nxt = true;
        }
        // pages of this tile: from the lookahead queue, else looked up now
        int blk, y;
        if (fv[0]) {
          blk = fb[0];
          y = fy[0];
        } else {
          const int raw = lane < NPG ? page_raw(cur, t, lane) : -2;
          blk = page_fix(cur, t, lane, raw, y);
        }
#pragma unroll
        for (int i = 0; i + 1 < D; ++i) fb[i] = fb[i + 1], fy[i] = fy[i + 1], fv[i] = fv[i + 1];
        // the tile D ahead (this item or the next): table entries requested now
        const int ta = t + D;
        const bool in_cur = ta < cur.ntiles;
        const WorkItem& ia = in_cur ? cur : nxt;
        const int tta = in_cur ? ta : ta - cur.ntiles;
        const bool av = in_cur || (nxt.b >= 0 && tta < nxt.ntiles);
        const int raw_a = (av && lane < NPG) ? page_raw(ia, tta, lane) : -2;
        if (lane == 0) TL(0, 1);
        if constexpr (F == kBF16) {
          // bf16 (nine boxes a tile): lane 0 issues the tile's boxes alone, from registers that
          // hold the tile's pages, so that the warp, which shares its sub-partition with busy
          // warps, spends few instructions a copy (decode 65.2 -> 64.0 us).  fp8 keeps the
          // warp-wide loop below: there the lean loop queued the next tiles' L2 prefetches
          // straight behind a full copy queue and the producer reached the next tile later
          // (0.864 -> 1.121 ms).
          int zq[8], yq[8];     // lane q < NPG resolved page q (NPG <= 8)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            zq[q] = __shfl_sync(0xFFFFFFFFu, blk, q);
            yq[q] = __shfl_sync(0xFFFFFFFFu, y, q);
          }
          if (lane == 0) {
#pragma unroll 1
            for (int b = 0; b < NB; ++b, ++pos) {
              const int slot = static_cast<int>(pos % R);
              if (C::kSlotCommits && pos >= R) {
                if (!mbar_wait(&empty[slot], static_cast<uint32_t>(pos / R - 1) & 1u, abort_flag)) {
                  ok = false;
                  break;
                }
              } else if (pos >= R) {
                const int tu = static_cast<int>((pos - R) / NB);     // tile that last used the slot
                if (tu != t_waited) {
                  if (!mbar_wait(&pv_done[tu & 1], static_cast<uint32_t>(tu >> 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                  }
                  t_waited = tu;
                }
              }
              if (F == kBF16 && b == 9) {
                mbar_arrive(&full[slot]);
                continue;
              }
              mbar_arrive_expect_tx(&full[slot], C::kSlot);
              if (b == 0 || b == NB - 1) TL(0, (b == 0 ? 1000 : 3000) + static_cast<int>((pos / NB) % 1000));
              const int x = (F == kFP8 && b == 4) ? 448 : 128 * b;
              uint8_t* dst = ring + slot * C::kSlot;
#pragma unroll
              for (int q = 0; q < 8; ++q)
                if (q < NPG) tma_load_3d(dst + q * p.BR * 128, &tm_kv, x, yq[q], zq[q], &full[slot]);
            }
          }
          // the warp goes on with lane 0's outcome
          ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
          pos = static_cast<int64_t>(__shfl_sync(0xFFFFFFFFu, static_cast<unsigned long long>(pos), 0));
          t_waited = __shfl_sync(0xFFFFFFFFu, t_waited, 0);
        } else {
#pragma unroll 1
          for (int b = 0; b < NB; ++b, ++pos) {
            const int slot = static_cast<int>(pos % R);
            if (C::kSlotCommits && pos >= R) {
              if (!warp_wait(&empty[slot], static_cast<uint32_t>(pos / R - 1) & 1u, abort_flag)) {
                ok = false;
                break;
              }
            } else if (pos >= R) {
              const int tu = static_cast<int>((pos - R) / NB);     // tile that last used the slot
              if (tu != t_waited) {
                if (!warp_wait(&pv_done[tu & 1], static_cast<uint32_t>(tu >> 1) & 1u, abort_flag)) {
                  ok = false;
                  break;
                }
                t_waited = tu;
              }
            }
            if (F == kBF16 && b == 9) {
              if (lane == 0) mbar_arrive(&full[slot]);
              continue;
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], C::kSlot);
            if (lane == 0 && (b == 0 || b == NB - 1)) TL(0, (b == 0 ? 1000 : 3000) + static_cast<int>((pos / NB) % 1000));
            __syncwarp();
            const int x = (F == kFP8 && b == 4) ? 448 : 128 * b;
            for (int q = 0; q < NPG; ++q) {
              const int z = __shfl_sync(0xFFFFFFFFu, blk, q);
              const int yy = __shfl_sync(0xFFFFFFFFu, y, q);
              if (lane == 0) tma_load_3d(ring + slot * C::kSlot + q * p.BR * 128, &tm_kv, x, yy, z, &full[slot]);
            }
          }
        }
        // finish the lookahead: queue its pages (and prefetch them into L2)
        {
          int ya = 0;
          const int ba = page_fix(ia, tta, lane, raw_a, ya);
          fb[D - 1] = ba;
          fy[D - 1] = ya;
          fv[D - 1] = av;
          for (int q = 0; q < NPG && av && C::kL2Pf; ++q) {
            const int z = __shfl_sync(0xFFFFFFFFu, ba, q);
            const int yy = __shfl_sync(0xFFFFFFFFu, ya, q);
            if (MLA_L2PF == 2) {
              if (z < p.num_blocks && lane == 0)
                bulk_prefetch_l2(p.kv + static_cast<int64_t>(z) * p.kv_blk_stride + static_cast<int64_t>(yy) * p.kv_ent_stride,
                                 static_cast<uint32_t>(p.BR * p.kv_ent_stride));
            } else if (z < p.num_blocks && lane < C::kNBQ) {
              tma_prefetch_3d(&tm_kv, (F == kFP8 && lane == 4) ? 448 : 128 * lane, yy, z);
            }
          }
        }
      }
      if (cur.ntiles > 0) {
        gt_next += cur.ntiles;
        gq = gt_next - 1;
      }
      if (!have_nxt) nxt = next_item(take_ticket());
      cur = nxt;
      have_nxt = false;
    }
    // end marker
    if (ok) {
      const int k = nitem % kItemDepth;
      if (nitem < kItemDepth || warp_wait(&item_empty[k], ((nitem / kItemDepth) - 1) & 1, abort_flag)) {
        if (lane == 0) {
          WorkItem e{};
          e.b = -1;
          items[k] = e;
          mbar_arrive(&item_full[k]);
        }
      }
    }
    // never leave copies in flight behind us
    if (lane == 0) {
      volatile int no_abort[2] = {0, 0};
      const int64_t first = pos > R ? pos - R : 0;
      for (int64_t q = first; q < pos; ++q) {
        const int slot = static_cast<int>(q % R);
        mbar_wait(&full[slot], static_cast<uint32_t>(q / R) & 1u, no_abort);
      }
      if (nq > 0) mbar_wait(q_full, (nq - 1) & 1, no_abort);
    }
    __syncwarp();
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (lane == 0 && errbits) set_device_error(p.err, errbits);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t ring_a = smem_u32(ring), q_a = smem_u32(qs), p_a = smem_u32(ps);
      const uint64_t dK0 = smem_desc(ring_a, 16, 1024, kSwizzle128B);
      const uint64_t dQ0 = smem_desc(q_a, 16, 1024, kSwizzle128B);
      const uint64_t dV0 = smem_desc(ring_a, C::kSlot, 1024, kSwizzle128B);
      constexpr uint32_t kPLbo = F == kBF16 ? NQ * 16 : NQ * 8;   // 8-key groups of P
      const uint64_t dP0 = smem_desc(p_a, kPLbo, 128, kSwizzleNone);
      constexpr uint32_t kIdQk = F == kBF16 ? idesc_f16(KM, NQ, 1, 1, 0, 0) : idesc_e4m3(KM, NQ, 0, 0);
      auto slot_of = [&](int gt, int b) -> int { return static_cast<int>((static_cast<int64_t>(gt) * NB + b) % R); };
      auto use_of = [&](int gt, int b) -> uint32_t {
        return static_cast<uint32_t>(((static_cast<int64_t>(gt) * NB + b) / R) & 1);
      };
      bool ok = true;
      int nit = 0, nq = 0, g = 0;
      // QK of global tile gt into S buffer gt & 1; returns false on a failed wait
      auto issue_pv = [&](int gt, bool first) -> bool {
        if (!mbar_wait(p_full, static_cast<uint32_t>(gt) & 1u, abort_flag)) return false;
        tc_fence_after();
        TL(2, 3);
        paged_issue_pv<C, F, NQ>(tmem, dV0, dP0, empty, gt, first);
        mma_commit(&pv_done[gt & 1]);
        TL(2, 4);
        return true;
      };
      // PV of tile pv_gt may be issued in the middle of a QK whose blocks are still landing
      // (the two write different accumulators)
      int pv_gt = -1;
      bool pv_first = false;
      auto issue_qk = [&](int gt, bool last) -> bool {
        const uint32_t dS = tmem + C::kTmemS + (gt & 1) * NQ;
        TL(2, 1);
        // the PV warp runs on its own: S[gt & 1] must have been read for tile gt - 2
        if (C::kPvSplit && gt >= 2 &&
            !mbar_wait(&s_free[gt & 1], static_cast<uint32_t>((gt - 2) >> 1) & 1u, abort_flag))
          return false;
        // ring position gt * NB + b: its slot and the parity of its use, walked per block
        int slot = slot_of(gt, 0);
        uint32_t use = use_of(gt, 0);
#pragma unroll 1
        for (int b = 0; b < NB; ++b) {
          if (b > 0 && ++slot == R) {
            slot = 0;
            use ^= 1u;
          }
          // wait for the block, but issue the pending PV as soon as its P is ready
          if (pv_gt >= 0 && !mbar_test_wait(&full[slot], use)) {
            const uint64_t t0 = globaltimer();
            for (uint32_t spin = 0;; ++spin) {
              if (mbar_test_wait(p_full, static_cast<uint32_t>(pv_gt) & 1u)) {
                if (!issue_pv(pv_gt, pv_first)) return false;
                pv_gt = -1;
                break;
              }
              if (mbar_try_wait_ns(&full[slot], use, 200)) break;
              if ((spin & 15u) == 15u && (*abort_flag || globaltimer() - t0 > kWaitNs)) break;   // the bounded wait below decides
            }
          }
          if (!mbar_wait(&full[slot], use, abort_flag)) return false;
          if (b == 0 || b == NB - 1) TL(2, (b == 0 ? 1000 : 2000) + gt % 1000);
          tc_fence_after();
          if (F == kBF16 && b == 9) {
            if (C::kSlotCommits) mbar_arrive(&empty[slot]);
            continue;
          }
          const uint64_t aK = desc_add(dK0, static_cast<uint32_t>(slot) * (C::kSlot >> 4));
          const uint64_t bQ = desc_add(dQ0, static_cast<uint32_t>(b) * (NQ * 128 >> 4));
          const uint32_t acc0 = b > 0 ? 1u : 0u;
          if (F == kBF16) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(dS, desc_add(aK, (kk * 32) >> 4), desc_add(bQ, (kk * 32) >> 4), kIdQk, kk > 0 ? 1u : acc0);
          } else {
            const int kk0 = (b == 4) ? 2 : 0;      // block 4 holds elements 448..575; 512.. are new
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (kk >= kk0)
                mma_f8_ss(dS, desc_add(aK, (kk * 32) >> 4), desc_add(bQ, (kk * 32) >> 4), kIdQk, kk > 0 ? 1u : acc0);
          }
        }
        mma_commit(&s_full[gt & 1]);
        if (C::kSlotCommits) mma_commit(&empty[slot_of(gt, C::kRope)]);
        TL(2, 2);
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
        if (C::kPvSplit) {
          for (int t = 0; t < it.ntiles && ok; ++t) ok = issue_qk(g + t, t == it.ntiles - 1);
        } else if (C::kOverlap) {
          ok = issue_qk(g, it.ntiles == 1);
          for (int t = 1; t < it.ntiles && ok; ++t) {
            pv_gt = g + t - 1;
            pv_first = (t == 1);
            ok = issue_qk(g + t, t == it.ntiles - 1);
            if (ok && pv_gt >= 0) ok = issue_pv(pv_gt, pv_first);
            pv_gt = -1;
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
      volatile int no_abort[2] = {0, 0};
      mbar_wait(fin, 0, no_abort);
    }
    __syncwarp();
  } else if (warp == C::kPvWarp) {
    // ------------------------------------------------------------------ PV issuer
    // A second MMA-issuing thread: PV(t) goes to the tensor cores as soon as P(t) is written,
    // in parallel with the next QK (a commit tracks the MMAs of its issuing thread).
    if (lane == 0) {
      const uint64_t dV0 = smem_desc(smem_u32(ring), C::kSlot, 1024, kSwizzle128B);
      constexpr uint32_t kPLbo = F == kBF16 ? NQ * 16 : NQ * 8;   // 8-key groups of P
      const uint64_t dP0 = smem_desc(smem_u32(ps), kPLbo, 128, kSwizzleNone);
      bool ok = true;
      int nit = 0, g = 0;
      while (ok) {
        const int k = nit % kItemDepth;
        if (!mbar_wait(&item_full[k], (nit / kItemDepth) & 1, abort_flag)) break;
        const WorkItem it = items[k];
        mbar_arrive(&item_empty[k]);
        ++nit;
        if (it.b < 0) break;
        for (int t = 0; t < it.ntiles && ok; ++t) {
          const int gt = g + t;
          const bool first = (t == 0);
          if (!mbar_wait(p_full, static_cast<uint32_t>(gt) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          TL(1, 1);
          paged_issue_pv<C, F, NQ>(tmem, dV0, dP0, empty, gt, first);
          mma_commit(&pv_done[gt & 1]);
          TL(1, 2);
        }
        g += it.ntiles;
      }
      mma_commit(fin_pv);
      volatile int no_abort[2] = {0, 0};
      mbar_wait(fin_pv, 0, no_abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    // Online softmax with a lazily moved reference max m (per column): p = 2^(s - m + kPExp)
    // stays below 2^(kTau + kPExp) as long as no logit exceeds m by more than kTau; only a
    // tile that does (a vote over all softmax threads) computes its exact column maxima,
    // moves m up to them and rescales O and the row sums by 2^(m_old - m_new).
    constexpr int NT = 32 * C::kSW;
    const int sw = warp - 2;
    const int quad = warp & 3;                  // TMEM lane quadrant of this warp
    const int c0 = (sw >> 2) * NC;              // first column of this thread
    const int row = quad * 32 + lane;           // TMEM lane: output column d of O^T
    const int krow = row;                       // key row of the tile (S^T lane)
    const int stid = tid - 64;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* red_m = red;                         // [2][NQ][4]
    float* red_l = red + 2 * NQ * 4;            // [NQ][4]
    // the reference max of every column (the same for all threads of a column half) lives in
    // shared memory rather than in 32 registers per thread; so does a rescale's factor
    float* mref = red + 3 * NQ * 4;             // [NQ]
    float* alph = mref + NQ;                    // [NQ]
    constexpr float kTau = F == kFP8 ? 4.f : 8.f;
    // row sums: per thread and column when registers allow (6 warps), else per warp and
    // column (lane % NC), reduced over the warp each tile
    constexpr bool kLReg = C::kSW == 4;
    constexpr int NL = kLReg ? NC : 1;
    constexpr float kPExp = F == kFP8 ? 4.f : 0.f;   // fp8: p carried as 2^4 p, at most 2^8 (e4m3 max 448)
    int nit = 0, g = 0;
    bool ok = true;
    while (ok) {
      const int k = nit % kItemDepth;
      bool w = warp_wait(&item_full[k], (nit / kItemDepth) & 1, abort_flag);
      const WorkItem it = items[k];
      ++nit;
      if (quad == 0 && (NC == 32 || lane < 16)) mref[c0 + (lane % NC)] = -CUDART_INF_F;
      if (!named_bar_and(1, NT, w)) break;
      if (it.b < 0) break;
      float l_part[NL];
#pragma unroll
      for (int c = 0; c < NL; ++c) l_part[c] = 0.f;
      const int cgb = it.g * NQ + c0;           // global column of this thread's column 0
      // logits of this thread's key for its columns, scaled and masked
      auto load_s = [&](float (&s)[NC], int gt, int t) {
        tmem_ld_n<NC>(tl + C::kTmemS + (gt & 1) * NQ + c0, s);
        tmem_ld_wait();
        const int kpos = it.k0 + t * KM + krow;
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
      };
      for (int t = 0; t < it.ntiles; ++t) {
        const int gt = g + t;
        w = warp_wait(&s_full[gt & 1], static_cast<uint32_t>(gt >> 1) & 1u, abort_flag);
        tc_fence_after();
        if (stid == 0) TL(3, 1);
        float s[NC];
        load_s(s, gt, t);
        const bool rv = it.k0 + t * KM + krow < it.k0 + it.n;
        // rows past the item never reach PV with stale contents
        if (!rv && c0 == 0) {
#pragma unroll 1
          for (int b = 0; b < (F == kBF16 ? 8 : 4); ++b) {
            uint4* dst = reinterpret_cast<uint4*>(
                ring + static_cast<int>((static_cast<int64_t>(gt) * NB + b) % R) * C::kSlot + krow * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          }
        }
        bool need = false;
#pragma unroll
        for (int c = 0; c < NC; c += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(mref + c0 + c);
          const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            need |= (s[c + u] > mm[u] + kTau) | ((mm[u] == -CUDART_INF_F) & (s[c + u] > -CUDART_INF_F));
        }
        if (stid == 0) TL(3, 10);
        // one barrier decides: nothing to do (common), or move the reference (or abort)
        if (C::kPvSplit) tc_fence_before();
        const bool rare = named_bar_or(1, NT, need || !w);
        if (C::kPvSplit && stid == 0) mbar_arrive(&s_free[gt & 1]);     // every thread has read S
        bool pv_waited = false;
        if (rare) {
          ok = named_bar_and(1, NT, w);
          if (!ok) break;
          float* rb = red_m + (gt & 1) * NQ * 4;
          {
            const float wm = warp_col_reduce<NC, true>(s, lane);
            if (NC == 32 || lane < 16) rb[(c0 + (lane % NC)) * 4 + quad] = wm;
          }
          named_bar_sync(1, NT);
          float mt_l;
          {
            const float4 q4 = reinterpret_cast<const float4*>(rb)[c0 + (lane % NC)];
            mt_l = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
          }
          // column (lane % NC): new reference and its factor, published once all have read the old
          const float mo_l = mref[c0 + (lane % NC)];
          const float mn_l = fmaxf(mo_l, mt_l);
          const float alpha_lane = (mo_l == -CUDART_INF_F) ? 0.f : ex2(mo_l - mn_l);
          const bool resc = __any_sync(0xFFFFFFFFu, mn_l != mo_l);
          named_bar_sync(1, NT);
          if (quad == 0 && (NC == 32 || lane < 16)) {
            mref[c0 + (lane % NC)] = mn_l;
            alph[c0 + (lane % NC)] = alpha_lane;
          }
          named_bar_sync(1, NT);
          float alpha[NC];
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            alpha[c] = alph[c0 + c];
            if (kLReg) l_part[kLReg ? c : 0] *= alpha[c];
          }
          if (!kLReg) l_part[0] *= alpha_lane;
          // O of the previous tiles moves to the new reference once PV of the last tile is done
          if (t > 0) {
            w = warp_wait(&pv_done[(gt - 1) & 1], static_cast<uint32_t>((gt - 1) >> 1) & 1u, abort_flag);
            tc_fence_after();
            pv_waited = true;
            if (w && resc) {
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
          load_s(s, gt, t);
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float mr = mref[c0 + c];
          const float mu = (mr == -CUDART_INF_F) ? 0.f : mr;
          s[c] = ex2(s[c] - mu + kPExp);
          if (kLReg) l_part[kLReg ? c : 0] += s[c];
        }
        if (stid == 0) TL(3, 2);
        if (t > 0 && !pv_waited) {
          w = warp_wait(&pv_done[(gt - 1) & 1], static_cast<uint32_t>((gt - 1) >> 1) & 1u, abort_flag);   // PV of the previous tile
          tc_fence_after();
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
            *reinterpret_cast<uint4*>(ps + (krow >> 3) * (NQ * 16) + (krow & 7) * 16 + ((c0 + c) >> 3) * 128) = v;
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
            const int off = (krow >> 3) * (NQ * 8) + (krow & 7) * 16 + ((c0 + c) >> 4) * 128;
            *reinterpret_cast<uint4*>(ps + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(ps + KM * NQ + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        // P of this warp's keys and columns is in place: one arrival per softmax warp, so PV
        // starts without a barrier of the group (a warp whose wait failed does not arrive; the
        // issuer's bounded wait then ends on the abort word)
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && w) mbar_arrive(p_full);
        if (stid == 0) TL(3, 3);
        ok = named_bar_and(1, NT, w);
        if (!ok) break;
        if (!kLReg) l_part[0] += warp_col_reduce<NC, false>(s, lane);   // while PV runs
      }
      if (!ok) break;
      // ---- epilogue: O / l and the LSE of every column of the item
      if (stid == 0) TL(3, 5);
      w = true;
      if (it.ntiles > 0) {
        w = warp_wait(&pv_done[(g + it.ntiles - 1) & 1], static_cast<uint32_t>((g + it.ntiles - 1) >> 1) & 1u, abort_flag);
        tc_fence_after();
      }
      g += it.ntiles;
      {
        float lw;
        if constexpr (kLReg) lw = warp_col_reduce<NC, false>(l_part, lane);
        else lw = l_part[0];
        if (NC == 32 || lane < 16) red_l[(c0 + (lane % NC)) * 4 + quad] = lw;
      }
      ok = named_bar_and(1, NT, w);
      if (!ok) break;
      // column (lane % NC): total row sum, 1 / l and the LSE; then 1 / l to every lane
      const int cl = lane % NC;
      float inv_l, lse_l;
      {
        const float4 q4 = reinterpret_cast<const float4*>(red_l)[c0 + cl];
        const float l = (q4.x + q4.y) + (q4.z + q4.w);
        const float m_l = mref[c0 + cl];
        const bool live = l > 0.f;
        inv_l = live ? __fdividef(p.out_scale, l) : 0.f;
        lse_l = live ? (m_l + __log2f(l) - kPExp) * 0.69314718055994531f : -CUDART_INF_F;
      }
      const bool final_out = (p.n_splits == 1);
      // (row, head) of column cg: row = b * q_len + cg / H, head = cg % H, so the flat index
      // row * H + head is b * q_len * H + cg
      const int64_t flat0 = static_cast<int64_t>(it.b) * p.q_len * p.H + cgb;
      const int ncol = min(NC, p.cols - cgb);
      const int64_t o_wrap = p.o_s0b - static_cast<int64_t>(p.H) * p.o_s1b;
      // O / l in slices of 16 columns (keeps the epilogue's live registers low)
#pragma unroll 1
      for (int jq = 0; jq < 4 * (NC / 16); ++jq) {
        const int j = jq / (NC / 16), cs = 16 * (jq % (NC / 16));
        float o[16];
        if (it.ntiles > 0) {
          tmem_ld16(tl + C::kTmemO + j * NQ + c0 + cs, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) o[c] = 0.f;
        }
        const int d = 128 * j + row;
        if (final_out) {
          // Running pointer over (token, head): the next column is the next head, or head 0 of
          // the next token after head H - 1 (no per-store index multiply).
          int h = (cgb + cs) % p.H;
          uint8_t* ptr = p.out + (static_cast<int64_t>(it.b) * p.q_len + (cgb + cs) / p.H) * p.o_s0b +
                         static_cast<int64_t>(h) * p.o_s1b + 2 * d;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float iv = __shfl_sync(0xFFFFFFFFu, inv_l, cs + c);
            if (cs + c < ncol) *reinterpret_cast<__nv_bfloat16*>(ptr) = __float2bfloat16_rn(o[c] * iv);
            ptr += p.o_s1b;
            if (++h == p.H) {
              h = 0;
              ptr += o_wrap;
            }
          }
        } else {
          float* dst = p.part_o + ((static_cast<int64_t>(it.s) * p.n_rows * p.H + flat0 + cs) * kLora + d);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float iv = __shfl_sync(0xFFFFFFFFu, inv_l, cs + c);
            if (cs + c < ncol) dst[static_cast<int64_t>(c) * kLora] = o[c] * iv;
          }
        }
      }
      if (row < 32 && (NC == 32 || lane < 16) && cl < ncol) {
        if (final_out) {
          if (p.lse) p.lse[flat0 + cl] = lse_l;
        } else {
          p.part_lse[static_cast<int64_t>(it.s) * p.n_rows * p.H + flat0 + cl] = lse_l;
        }
      }
      tc_fence_before();
      named_bar_sync(1, NT);
      if (stid == 0) mbar_arrive(&item_empty[k]);
      if (stid == 0) TL(3, 6);
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
