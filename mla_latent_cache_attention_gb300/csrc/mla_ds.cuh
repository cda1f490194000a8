// mla_ds.cuh -- MLA over the 656-byte fp8_ds_mla record: the sparse (CSR-indexed) forward and
// the paged decode / spec-verify.
//
// What it computes ("vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla", flydsl_sparse_mla_fp8ds_fwd:
// the sparse forward over CSR key lists, masked negative indices, empty row -> 0 / -inf,
// natural-log lse, and the 656-byte record; "vllm.models.kimi_k3.nvidia.specialized_decode.
// cutedsl.mla.prepared", trtllm_decode: the paged decode over the same records): a record holds
// 512 e4m3 codes of kv_c_normed in four 128-wide tiles with one fp32 scale each, then 64 bf16
// of k_pe.  The key is k = [s_j * code_j (j = 0..3) | k_pe], the value its first 512 entries; the
// logit of query q is softmax_scale * q . k.
//
// How (GB300 design, exact up to fp32 accumulation):
//   * QK on the tensor cores directly on the e4m3 codes (kind::f8f6f4): the bf16 query of
//     every column c is split into two e4m3 terms hi + lo of 2^e_c q (an e4m3 holds 4
//     significant bits, a bf16 8, so hi + lo carries q exactly wherever 2^e_c |q| >= 2^-2),
//     stacked as 2 x 16 columns of the B operand.  Each key tile j accumulates separately
//     (S_j, 32 TMEM columns) and the softmax forms s = 2^-e_c sum_j s_j (S_j,hi + S_j,lo) +
//     S_rope, so the per-key scale is applied in fp32.  k_pe . q_pe runs as a bf16 MMA.
//   * PV on the e4m3 codes as well: O_j^T = V_j^T P_j with P_j = p * s_j * r_j, one P per value
//     tile so that each key's scale multiplies its own term, as four e5m2 terms (stacked
//     along N, 16 columns each; e4m3 codes x e5m2 weights): the first is P_j rounded to
//     nearest e5m2 from fp32, and the exact rest (at most 2^-3 of P_j) is rounded once to
//     f16 and split on its bits (an e5m2 is the upper byte of an f16: two terms keep 3
//     significant bits each of what is left and the last rounds the rest), so the four carry
//     P_j to about 2^-12 relative -- the outputs cancel terms up to 448 times a scale, and a
//     plain f16 P (2^-11) measured up to 1.1 times the tolerance on random shapes -- and
//     e5m2 reaches down to 2^-16, which keeps the many small weights of a long row from being
//     lost under an e4m3 floor of 2^-9.  r_j is a power of two kept per item so
//     that s_j r_j <= 1; when a later key needs a smaller r_j, O_j is rescaled by the (exact)
//     ratio.
//   * Online softmax with a lazily moved reference max, as in the page kernel.
//   * Paged source: TMA page boxes (four code tiles, k_pe, and the scales through a second,
//     unswizzled map) into a two-tile ring.  Sparse source: eight gather warps load each
//     record with 16-byte vector loads (a record is 41 of them) and store it in the same
//     layout; masked or out-of-range indices store zeros and a row flag.
//   * Roles hand over through mbarriers, each waited with a time limit: a gathered tile
//     completes one barrier (one arrival per gather warp, after all its stores); S is released
//     per softmax warp as soon as its TMEM loads are done; P_j completes a barrier of its own
//     (one arrival per softmax warp), so the PV of value tile j runs while the later P_j are
//     written.
//
// Warps: 0 scheduler (+ TMA producer for pages; + PV issuer for the sparse source), 1 QK issuer
// (TMEM owner), 2..5 softmax + query preparation + epilogue, then 6 PV issuer (pages) or
// 6..13 gather (sparse).
#pragma once
#include "mla_paged_tma.cuh"

namespace mla {

struct DsParams {
  const uint8_t* q;               // bf16 [rows][H][>=576]
  int64_t q_s0b, q_s1b;
  int H, q_len, B, G, cols;       // B requests (sparse: query rows), G groups of 16 columns
  // sparse source
  const uint8_t* records;
  int64_t rec_stride, num_records;
  const int32_t* indptr;
  const int32_t* indices;
  int has_invalid;
  // paged source
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;
  int num_blocks, block_size, BR;
  int chunk, n_splits, n_items, n_rows;
  float sig2;                     // softmax scale * log2(e)
  uint8_t* out;
  int64_t o_s0b, o_s1b;
  float* lse;
  float* part_o;
  float* part_lse;
  uint32_t* sched;
  uint32_t* err;
  int partial;                    // write fp32 partials (part_o / part_lse) instead of out / lse
  int split_base;                 // sparse: partial index of this launch's split 0
};

template <bool kSparse>
struct DsCfg {
  static constexpr int NQ = 16, NB = 5, R = 10;        // a tile is 5 ring slots; the ring holds two
  static constexpr int kGatherWarps = kSparse ? 8 : 0;
  // PV has its own issuing thread: pages, warp 6 (after the softmax warps); sparse, lane 0 of
  // the scheduler warp (a 15th warp beside the gather warps cost more than it saved)
  static constexpr int kPvWarp = kSparse ? -1 : 6;
  static constexpr int kThreads = 192 + 32 * kGatherWarps + (kSparse ? 0 : 32);
  static constexpr int kRing = 0;
  static constexpr int kScale = kRing + R * kSlotBytes;          // [2][128] float4
  static constexpr int kQ = kScale + 2 * kTile * 16;              // 4 x (32 rows x 128 B) hi/lo + 16 x 128 B rope
  static constexpr int kQRope = kQ + 4 * 32 * 128;
  static constexpr int kP = kQRope + NQ * 128;                    // 4 x (128 keys x 64 B)
  static constexpr int kRed = kP + 4 * kTile * 64;                // [2][16][4] max, [16][4] sum, [4][4] scale max
  static constexpr int kColF = kRed + (3 * NQ * 4 + 16) * 4;      // [16] 2^-e_c
  static constexpr int kMref = kColF + NQ * 4;                    // [4 warps][16] reference max, per warp
  static constexpr int kAlph = kMref + 4 * NQ * 4;                // [4 warps][16] rescale factors, per warp
  static constexpr int kRj = kAlph + 4 * NQ * 4;                  // [4 warps][8] r_j, O_j rescale ratios
  static constexpr int kValid = kRj + 4 * 8 * 4;                  // [2][128] row flags (sparse)
  static constexpr int kItems = kValid + 2 * kTile;
  static constexpr int kBar = kItems + kItemDepth * 32;
  // + ring_free[2] and xitem_full[kItemDepth] of the CTA-pair kernel
  // + p_full[4] (one per value tile)
  static constexpr int kNumBars = R + 8 + 2 * kItemDepth + 2 + kItemDepth + 4;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 16 + 8 * 8;   // TMEM slot, abort word, cluster CTAs' ring positions
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= kSmemLimit, "shared memory budget");
  static constexpr int kS = 0;                                    // S (144 columns): S_j at 32 j, rope at 128
  static constexpr int kTmemO = 160;                              // O_j at kTmemO + 64 j (4 terms x 16 columns)
  static constexpr int kTmemCols = 512;
};

__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }   // e in [-126, 127]

// Two floats rounded to nearest even e5m2 (saturating), a in the low byte, and back.
__device__ __forceinline__ uint32_t e5m2x2_rn(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E5M2));
}
__device__ __forceinline__ float2 e5m2x2_to_float2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E5M2);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// 2^e with e the largest integer such that a * 2^e <= 448 (a > 0 finite), clamped to the
// normal range.
__device__ __forceinline__ int e4m3_fit_exponent(float a) {
  if (!(a > 0.f)) return 0;
  int e = 8 - (static_cast<int>((__float_as_uint(a) >> 23) & 0xFF) - 127);   // a * 2^e in [256, 512)
  e = max(min(e, 126), -126);
  while (e > -126 && a * pow2i(e) > 448.f) --e;
  while (e < 126 && a * pow2i(e + 1) <= 448.f) ++e;
  return e;
}

// PV of value tile j of tile gt: O_j (+)= V_j^T P_j (V_j: ring slot j of the tile's half of
// the ring; P_j: 128 keys x 64 weights).  Issued per value tile as soon as its P_j is written,
// so the four PV blocks overlap the softmax's writing of the later P_j.  The descriptors
// advance by 32-bit adds: the issuing thread shares its sub-partition with busy warps, and
// fewer instructions per MMA measured faster.
template <int NB>
__device__ __forceinline__ void ds_issue_pv_block(uint32_t tmem_o, uint64_t dV0, uint64_t dP0, uint32_t id, int gt,
                                                  int j, bool first) {
  const uint64_t aV = desc_add(dV0, (((gt & 1) * NB + j) * kSlotBytes) >> 4);
  const uint64_t bP = desc_add(dP0, (j * kTile * 64) >> 4);
  const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_f8_ss(tmem_o + 64 * j, desc_add(aV, (kk * 4096) >> 4), desc_add(bP, (kk * 2048) >> 4), id, kk > 0 ? 1u : acc0);
}

// kCl = 2, 3 or 6 (paged source only): the kernel runs as clusters of kCl CTAs.  The CTAs of a
// cluster take the same item (request, split) for kCl adjacent column groups: the cluster's
// first CTA takes the tickets and passes each item to the others through a mailbox in its
// shared memory; each CTA issues 1/kCl of every tile's page boxes with cluster multicast, so
// every ring receives the whole tile while each SM's copy engine issues a share of it and L2
// serves each key once per cluster; a ring slot is reused only once every CTA's PV of the tile
// before has finished with it (a multicast commit into a kCl-arrival barrier of each CTA).
template <bool kSparse, int kCl>
__global__ void __launch_bounds__(DsCfg<kSparse>::kThreads, 1)
    mla_ds_kernel(const __grid_constant__ DsParams p, const __grid_constant__ CUtensorMap tm_kv,
                  const __grid_constant__ CUtensorMap tm_sc) {
  static_assert(kCl == 1 || ((kCl == 2 || kCl == 3 || kCl == 6) && !kSparse), "clusters serve the paged source");
  using C = DsCfg<kSparse>;
  static_assert(C::kItems % 16 == 0 && C::kMisc % 8 == 0, "queue slots are read as 16-byte words");
  constexpr int R = C::R, NB = C::NB, NQ = C::NQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + C::kRing;
  float4* scl = reinterpret_cast<float4*>(smem + C::kScale);      // [2][128]
  uint8_t* qs = smem + C::kQ;
  uint8_t* qr = smem + C::kQRope;
  uint8_t* ps = smem + C::kP;
  float* red = reinterpret_cast<float*>(smem + C::kRed);
  float* colf = reinterpret_cast<float*>(smem + C::kColF);
  uint8_t* vrow = smem + C::kValid;                                 // [2][128]
  WorkItem* items = reinterpret_cast<WorkItem*>(smem + C::kItems);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* full = bars;                  // [R] slot data landed (TMA bytes; sparse: the gather warps complete a tile's first)
  uint64_t* s_full = bars + R;            // [2]
  uint64_t* pv_done = bars + R + 2;       // [2]
  uint64_t* q_full = bars + R + 4;
  uint64_t* fin = bars + R + 5;
  uint64_t* s_free = bars + R + 6;        // the softmax warps have read S (four arrivals)
  uint64_t* item_full = bars + R + 7;
  uint64_t* item_empty = item_full + kItemDepth;
  uint64_t* fin_pv = item_empty + kItemDepth;
  uint64_t* ring_free = fin_pv + 1;       // [2] cluster: every CTA's PV of the tile is done
  uint64_t* xitem_full = ring_free + 2;   // [kItemDepth] cluster: the first CTA's item k is posted
  // [4] P_j of the tile is written (one arrival per softmax warp): PV of value tile j may go
  uint64_t* p_full = xitem_full + kItemDepth;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);
  int64_t* cl_pos = reinterpret_cast<int64_t*>(smem + C::kMisc + 16);   // [kCl] cluster: positions each producer issued
  const uint32_t crank = kCl > 1 ? cluster_ctarank() : 0u;
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << kCl) - 1u);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  TL_DECL;

  // the split-K merge may be scheduled now; it waits for this grid to complete
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < R; ++i) mbar_init(&full[i], kSparse ? C::kGatherWarps : 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&pv_done[i], 1);
    }
    for (int j = 0; j < 4; ++j) mbar_init(&p_full[j], 4);
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    mbar_init(fin_pv, 1);
    mbar_init(s_free, 4);     // one arrival per softmax warp
    for (int k = 0; k < kItemDepth; ++k) {
      mbar_init(&item_full[k], 1);
      // the cluster's first CTA also waits for the other producers to have read item k
      mbar_init(&item_empty[k], 3 + C::kGatherWarps + ((kCl > 1 && crank == 0) ? kCl - 1 : 0));
      mbar_init(&xitem_full[k], 1);
    }
    mbar_init(&ring_free[0], kCl);
    mbar_init(&ring_free[1], kCl);
    *abort_flag = 0;
    abort_flag[1] = 0;
    for (int r = 0; r < 8; ++r) cl_pos[r] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // cluster: every CTA's barriers exist before any CTA signals another or copies into it
  if (kCl > 1) cluster_sync();
  const uint32_t tmem = *tmem_slot;
  // launched as a programmatic dependent of the previous kernel in the stream: the setup above
  // overlaps that kernel's tail, and its writes (a decode epilogue's query and cache entry, the
  // scheduler reset) are visible past this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // items: (split s, request / row b, column group g)
  // cluster: an item covers kCl adjacent column groups, the one of CTA r being kCl * g' + r
  auto decode = [&](int item, WorkItem& it) -> bool {     // false: an empty split (skipped)
    it.b = -1;
    if (item >= p.n_items) return true;
    const int Gc = (p.G + kCl - 1) / kCl;
    const int bg = p.B * Gc;
    it.s = item / bg;
    it.b = (item % bg) / Gc;
    it.g = (item % Gc) * kCl + static_cast<int>(crank);
    it.pad = 0;
    if (kSparse) {
      // split s of the row: keys [s c, (s + 1) c) of its list, c = ceil(n / n_splits) rounded
      // up to whole tiles; every split runs (an empty one writes a 0 / -inf partial)
      const int b0 = p.indptr[it.b], nr = max(p.indptr[it.b + 1] - b0, 0);
      const int c = p.n_splits > 1 ? ((nr + p.n_splits - 1) / p.n_splits + kTile - 1) / kTile * kTile : nr;
      const int s0 = min(it.s * c, nr);
      it.k0 = b0 + s0;
      it.n = min(c, nr - s0);
      it.L = it.k0 + it.n;
      it.s += p.split_base;
    } else {
      it.L = max(p.seq_lens[it.b], 0);
      it.k0 = it.s * p.chunk;
      it.n = min(max(it.L - it.k0, 0), p.chunk);
    }
    it.ntiles = (it.n + kTile - 1) / kTile;
    return kSparse || it.n > 0 || p.n_splits == 1;
  };

  if (warp == 0 && kSparse) {
    // ------------------------------------------------------------------ scheduler + PV issuer
    // Sparse source: warp 0 has no pages to load, so its lane 0 both hands out work items and
    // issues PV(t) as soon as P(t) is written (a second MMA-issuing thread beside the QK warp;
    // a commit tracks its issuing thread).  It polls both sides and never blocks on one.
    if (lane == 0) {
      int stride_k = 0;
      auto take = [&]() -> int {
        const int item = p.sched ? static_cast<int>(atomicAdd(p.sched, 1u)) : static_cast<int>(blockIdx.x + stride_k * gridDim.x);
        ++stride_k;
        return item;
      };
      auto next_item = [&]() -> WorkItem {
        WorkItem it{};
        while (!decode(take(), it)) {
        }
        return it;
      };
      const uint64_t dV0 = smem_desc(smem_u32(ring), kSlotBytes, 1024, kSwizzle128B);
      const uint64_t dP0 = smem_desc(smem_u32(ps), 512, 128, kSwizzleNone);
      constexpr uint32_t kIdPv = idesc_e4m3(128, 64, 1, 1) | (1u << 10);   // B (weights) in e5m2
      WorkItem cur = next_item(), pit{};
      int npush = 0, npv = 0, pv_t = 0, pv_g = 0, pv_j = 0;
      bool push_done = false, have = false;
      uint64_t t_last = globaltimer();
      for (;;) {
        bool prog = false;
        if (!push_done) {
          const int k = npush % kItemDepth;
          if (npush < kItemDepth || mbar_test_wait(&item_empty[k], static_cast<uint32_t>((npush / kItemDepth) - 1) & 1u)) {
            items[k] = cur;
            mbar_arrive(&item_full[k]);
            ++npush;
            if (cur.b < 0)
              push_done = true;
            else
              cur = next_item();
            prog = true;
          }
        }
        if (!have) {
          const int k = npv % kItemDepth;
          if (npv < npush && mbar_test_wait(&item_full[k], static_cast<uint32_t>(npv / kItemDepth) & 1u)) {
            pit = items[k];
            mbar_arrive(&item_empty[k]);
            ++npv;
            prog = true;
            if (pit.b < 0) break;
            have = true;
            pv_t = 0;
          }
        } else if (pv_t < pit.ntiles) {
          const int gt = pv_g + pv_t;
          if (mbar_test_wait(&p_full[pv_j], static_cast<uint32_t>(gt) & 1u)) {
            tc_fence_after();
            if (pv_j == 0) TL(0, 1);
            ds_issue_pv_block<NB>(tmem + C::kTmemO, dV0, dP0, kIdPv, gt, pv_j, pv_t == 0);
            if (++pv_j == 4) {
              pv_j = 0;
              mma_commit(&pv_done[gt & 1]);
              TL(0, 2);
              ++pv_t;
            }
            prog = true;
          }
        } else {
          pv_g += pit.ntiles;
          have = false;
          prog = true;
        }
        if (prog) {
          t_last = globaltimer();
        } else {
          if (*abort_flag) break;
          if (globaltimer() - t_last > kWaitNs) {
            *abort_flag = 2;
            break;
          }
          if (have && pv_t < pit.ntiles) (void)mbar_try_wait_ns(&p_full[pv_j], static_cast<uint32_t>(pv_g + pv_t) & 1u, 500);
        }
      }
      mma_commit(fin_pv);
      volatile int no_abort[2] = {0, 0};
      mbar_wait(fin_pv, 0, no_abort);
    }
    __syncwarp();
  } else if (!kSparse && warp == 0) {
    // ------------------------------------------------------------------ scheduler / page producer
    uint32_t errbits = 0;
    int nitem = 0, stride_k = 0, gt_next = 0;
    bool ok = true;
    // tickets: one counter per launch (or a static stride when there is none); a cluster's
    // tickets are taken by its first CTA
    const int unit = static_cast<int>(blockIdx.x) / kCl, n_units = static_cast<int>(gridDim.x) / kCl;
    auto take_ticket = [&]() -> int {
      int item = 0;
      if (lane == 0) item = p.sched ? static_cast<int>(atomicAdd(p.sched, 1u)) : unit + stride_k * n_units;
      ++stride_k;
      return __shfl_sync(0xFFFFFFFFu, item, 0);
    };
    // the next item of this CTA (false: a wait ran out).  The cluster's other CTAs read item
    // nitem from the first CTA's queue slot once it is posted, then release that slot.
    auto fetch = [&](WorkItem& it) -> bool {
      if (kCl == 1 || crank == 0) {
        while (!decode(take_ticket(), it)) {
        }
        return true;
      }
      const int k = nitem % kItemDepth;
      if (!warp_wait_cl(&xitem_full[k], static_cast<uint32_t>(nitem / kItemDepth) & 1u, abort_flag)) return false;
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
      if (lane == 0) {
        const uint32_t src = mapa_shared(&items[k], 0);
        v0 = ld_cluster_v4(src);
        v1 = ld_cluster_v4(src + 16);
        mbar_arrive_remote(mapa_shared(&item_empty[k], 0));
      }
      const uint32_t f[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t g[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = __shfl_sync(0xFFFFFFFFu, f[i], 0);
      static_assert(sizeof(WorkItem) == 32, "a queue slot is two 16-byte words");
      memcpy(&it, g, sizeof(WorkItem));
      if (it.b >= 0) it.g += static_cast<int>(crank);
      return true;
    };
    // post item `it` to this CTA's roles (and, from a cluster's first CTA, to the others)
    auto push = [&](const WorkItem& it) -> bool {
      const int k = nitem % kItemDepth;
      if (nitem >= kItemDepth) {
        const uint32_t par = static_cast<uint32_t>((nitem / kItemDepth) - 1) & 1u;
        const bool w = (kCl > 1 && crank == 0) ? warp_wait_cl(&item_empty[k], par, abort_flag)
                                               : warp_wait(&item_empty[k], par, abort_flag);
        if (!w) return false;
      }
      if (lane == 0) {
        items[k] = it;
        mbar_arrive(&item_full[k]);
        if (kCl > 1 && crank == 0)
          for (int r = 1; r < kCl; ++r) mbar_arrive_remote(mapa_shared(&xitem_full[k], static_cast<uint32_t>(r)));
      }
      ++nitem;
      return true;
    };
    const int NPG = kTile / max(p.BR, 1);
    int64_t pos = 0;
    int t_waited = -1;
    WorkItem cur{};
    ok = fetch(cur);
    while (ok && cur.b >= 0) {
      if (!push(cur)) {
        ok = false;
        break;
      }
      {
        for (int t = 0; t < cur.ntiles && ok; ++t) {
          const int gt = gt_next + t;
          int blk = p.num_blocks, y = 0;
          if (lane < NPG) {
            const int kp = cur.k0 + t * kTile + lane * p.BR;
            if (kp < cur.k0 + cur.n) {
              const int id = p.block_table[static_cast<int64_t>(cur.b) * p.bt_stride + kp / p.block_size];
              if (id >= 0 && id < p.num_blocks) {
                blk = id;
                y = kp % p.block_size;
              } else {
                errbits |= 2u;
              }
            }
          }
          // the two-tile ring: tile gt reuses the slots of tile gt - 2 (a cluster: in every CTA)
          if (lane == 0) TL(0, 1);
          if (gt >= 2 && gt - 2 != t_waited) {
            const uint32_t par = static_cast<uint32_t>((gt - 2) >> 1) & 1u;
            if (!(kCl > 1 ? warp_wait_cl(&ring_free[gt & 1], par, abort_flag)
                          : warp_wait(&pv_done[gt & 1], par, abort_flag))) {
              ok = false;
              break;
            }
            t_waited = gt - 2;
          }
          if (lane == 0) TL(0, 2);
#pragma unroll 1
          for (int b = 0; b < NB; ++b, ++pos) {
            const int slot = static_cast<int>(pos % R);
            // the slot's whole tile lands here (a cluster: a share from each CTA's boxes)
            const uint32_t bytes = kSlotBytes + (b == NB - 1 ? static_cast<uint32_t>(kTile * 16) : 0u);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], bytes);
            __syncwarp();
            const int x = (b == NB - 1) ? 528 : 128 * b;
            for (int q = 0; q < NPG; ++q) {
              const int z = __shfl_sync(0xFFFFFFFFu, blk, q);
              const int yy = __shfl_sync(0xFFFFFFFFu, y, q);
              if (lane == 0 && (kCl == 1 || (b * NPG + q) % kCl == static_cast<int>(crank))) {
                uint8_t* dk = ring + slot * kSlotBytes + q * p.BR * 128;
                uint8_t* ds = reinterpret_cast<uint8_t*>(scl + (gt & 1) * kTile) + q * p.BR * 16;
                if (kCl > 1) {
                  tma_load_3d_mc(dk, &tm_kv, x, yy, z, &full[slot], kMask);
                  if (b == NB - 1) tma_load_3d_mc(ds, &tm_sc, 512, yy, z, &full[slot], kMask);
                } else {
                  tma_load_3d(dk, &tm_kv, x, yy, z, &full[slot]);
                  if (b == NB - 1) tma_load_3d(ds, &tm_sc, 512, yy, z, &full[slot]);
                }
              }
            }
          }
        }
      }
      gt_next += cur.ntiles;
      if (ok) ok = fetch(cur);
    }
    if (ok) {
      WorkItem e{};
      e.b = -1;
      (void)push(e);
    }
    if (kCl > 1) {
      // every CTA's drain learns the positions this producer issued (it runs after the final
      // cluster barrier, when no producer issues any more)
      if (lane == 0)
        for (int r = 0; r < kCl; ++r)
          st_cluster_u64(mapa_shared(&cl_pos[crank], static_cast<uint32_t>(r)), static_cast<uint64_t>(pos));
    } else if (lane == 0) {     // never leave copies in flight behind us
      volatile int no_abort[2] = {0, 0};
      const int64_t first = pos > R ? pos - R : 0;
      for (int64_t q = first; q < pos; ++q) mbar_wait(&full[q % R], static_cast<uint32_t>(q / R) & 1u, no_abort);
    }
    __syncwarp();
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (lane == 0 && errbits) set_device_error(p.err, errbits);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ QK issuer (TMEM owner)
    if (lane == 0) {
      const uint32_t ring_a = smem_u32(ring), q_a = smem_u32(qs), qr_a = smem_u32(qr);
      const uint64_t dK0 = smem_desc(ring_a, 16, 1024, kSwizzle128B);
      const uint64_t dQ0 = smem_desc(q_a, 16, 1024, kSwizzle128B);
      const uint64_t dQr = smem_desc(qr_a, 16, 1024, kSwizzle128B);
      // QK only; PV goes to its own issuing thread
      constexpr uint32_t kIdNope = idesc_e4m3(128, 32, 0, 0);
      constexpr uint32_t kIdRope = idesc_f16(128, 16, 1, 1, 0, 0);
      auto slot_of = [&](int gt, int b) -> int { return (gt & 1) * NB + b; };
      auto issue_qk = [&](int gt) -> bool {
        TL(2, 1);
        // one S buffer: the softmax of the previous tile must have read it
        if (gt > 0 && !mbar_wait(s_free, static_cast<uint32_t>(gt - 1) & 1u, abort_flag)) return false;
        tc_fence_after();
        TL(2, 5);
        const uint32_t dS = tmem + C::kS;
        if (kSparse) {
          // the gather warps arrive on the tile's first slot barrier only, after all their
          // stores to the tile: one wait covers the five slots (fewer instructions for a thread
          // that shares its sub-partition with busy warps).  The MMAs stay in a per-slot loop:
          // issuing all 20 in a straight line measured slower.
          const int s0 = (gt & 1) * NB;
          if (!mbar_wait(&full[s0], static_cast<uint32_t>(gt >> 1) & 1u, abort_flag)) return false;
          tc_fence_after();
#pragma unroll 1
          for (int b = 0; b < NB; ++b) {
            const uint64_t aK = dK0 + (((s0 + b) * kSlotBytes) >> 4);
            if (b < 4) {
              const uint64_t bQ = dQ0 + ((b * 32 * 128) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f8_ss(dS + 32 * b, aK + ((kk * 32) >> 4), bQ + ((kk * 32) >> 4), kIdNope, kk > 0 ? 1u : 0u);
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ss(dS + 128, aK + ((kk * 32) >> 4), dQr + ((kk * 32) >> 4), kIdRope, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&s_full[0]);
          TL(2, 2);
          return true;
        }
#pragma unroll 1
        for (int b = 0; b < NB; ++b) {
          const int slot = slot_of(gt, b);
          if (!mbar_wait(&full[slot], static_cast<uint32_t>(gt >> 1) & 1u, abort_flag)) return false;
          tc_fence_after();
          const uint64_t aK = dK0 + ((slot * kSlotBytes) >> 4);
          if (b < 4) {
            const uint64_t bQ = dQ0 + ((b * 32 * 128) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8_ss(dS + 32 * b, aK + ((kk * 32) >> 4), bQ + ((kk * 32) >> 4), kIdNope, kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(dS + 128, aK + ((kk * 32) >> 4), dQr + ((kk * 32) >> 4), kIdRope, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(&s_full[0]);
        TL(2, 2);
        return true;
      };
      bool ok = true;
      int nit = 0, nq = 0, g = 0;
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
        for (int t = 0; t < it.ntiles && ok; ++t) ok = issue_qk(g + t);
        g += it.ntiles;
      }
      mma_commit(fin);
      volatile int no_abort[2] = {0, 0};
      mbar_wait(fin, 0, no_abort);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------------ softmax, query, epilogue
    constexpr int NT = 128;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int stid = tid - 64;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* red_m = red;                 // [2][16][4]
    float* red_l = red + 2 * NQ * 4;    // [16][4]
    float* red_s = red + 3 * NQ * 4;    // [4 warps][4 tiles] scale maxima
    // p = 2^(s - m_ref + kPExp) <= 2^(kTau + kPExp) = 2^14 keeps P_j = p s_j r_j inside f16
    // and e5m2 (both past 2^15), and the lazy reference moves only on a jump of kTau
    constexpr float kTau = 10.f, kPExp = 4.f;
    constexpr int kOB = kSparse ? 32 : 64;      // TMEM columns per O-rescale round trip (registers)
    // The query of item qi into the query buffer (every softmax thread; ends with the group
    // barrier and the q_full arrival): thread (c = stid / 8, part = stid % 8) handles elements
    // 64 part .. +63 of column c; hi / lo e4m3 of 2^e_c q into rows c / 16 + c, k_pe as it is
    auto prep_query = [&](const WorkItem& qi) {
      const int c = stid >> 3, part = stid & 7;
      const int cg = qi.g * NQ + c;
      const bool live = cg < p.cols;
      const uint8_t* qrow = live ? p.q + (static_cast<int64_t>(qi.b) * p.q_len + cg / p.H) * p.q_s0b + (cg % p.H) * p.q_s1b
                                 : nullptr;
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = live ? *reinterpret_cast<const uint4*>(qrow + part * 128 + 16 * i) : make_uint4(0, 0, 0, 0);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          amax = fmaxf(amax, fabsf(__uint_as_float(wv[u] << 16)));
          amax = fmaxf(amax, fabsf(__uint_as_float(wv[u] & 0xFFFF0000u)));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
      const int e = e4m3_fit_exponent(amax);
      const float sc = pow2i(e);
      if (part == 0) colf[c] = pow2i(-e);
      // 64 elements -> 64 hi bytes + 64 lo bytes at block part / 2, byte (part & 1) * 64
      const int blk = part >> 1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {     // 16 elements per 16-byte output chunk
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 a = v[2 * i + (u >> 1)];
          const uint32_t w0 = (u & 1) ? a.z : a.x, w1 = (u & 1) ? a.w : a.y;
          const float x0 = __uint_as_float(w0 << 16) * sc, x1 = __uint_as_float(w0 & 0xFFFF0000u) * sc;
          const float x2 = __uint_as_float(w1 << 16) * sc, x3 = __uint_as_float(w1 & 0xFFFF0000u) * sc;
          const uint32_t h01 = e4m3x2_sat(x0, x1), h23 = e4m3x2_sat(x2, x3);
          const float2 f01 = e4m3x2_to_float2(h01), f23 = e4m3x2_to_float2(h23);
          hw[u] = h01 | (h23 << 16);
          lw[u] = e4m3x2_sat(x0 - f01.x, x1 - f01.y) | (e4m3x2_sat(x2 - f23.x, x3 - f23.y) << 16);
        }
        const int chunk = (part & 1) * 4 + i;
        uint8_t* base = qs + blk * (32 * 128);
        *reinterpret_cast<uint4*>(base + sw128(c, chunk)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(base + sw128(16 + c, chunk)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      // k_pe part: 128 bytes per column, one 16-byte chunk per thread
      const uint4 rv = live ? *reinterpret_cast<const uint4*>(qrow + 1024 + 16 * part) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(qr + sw128(c, part)) = rv;
      fence_proxy_async_smem();
      named_bar_sync(1, NT);
      if (stid == 0) mbar_arrive(q_full);
    };
    int nit = 0, g = 0;
    bool ok = true;
    bool q_ready = false;      // the query of the next item was prepared ahead of the epilogue
    while (ok) {
      const int k = nit % kItemDepth;
      bool w = warp_wait(&item_full[k], (nit / kItemDepth) & 1, abort_flag);
      const WorkItem& it = items[k];     // read in place (registers): the slot is ours until item_empty
      ++nit;
      if (!named_bar_and(1, NT, w)) break;
      if (it.b < 0) break;
      const int cgb = it.g * NQ;     // first global column of the item
      if (it.ntiles > 0 && !q_ready) prep_query(it);
      q_ready = false;
      // the column reference maxima and rescale factors are the same for every thread: one
      // copy per warp in shared memory keeps them out of the registers
      float* mref = reinterpret_cast<float*>(smem + C::kMref) + quad * NQ;
      float* alph = reinterpret_cast<float*>(smem + C::kAlph) + quad * NQ;
      if (lane < NQ) mref[lane] = -CUDART_INF_F;
      __syncwarp();
      float l_part[NQ];
#pragma unroll
      for (int c = 0; c < NQ; ++c) l_part[c] = 0.f;
      float* rj = reinterpret_cast<float*>(smem + C::kRj) + quad * 8;   // per value tile: P_j = p s_j r_j (0: not set yet)
      float* ratio = rj + 4;
      if (lane < 4) rj[lane] = 0.f;
      __syncwarp();
      for (int t = 0; t < it.ntiles; ++t) {
        const int gt = g + t;
        w = warp_wait(&s_full[0], static_cast<uint32_t>(gt) & 1u, abort_flag);
        tc_fence_after();
        if (stid == 0) TL(3, 1);
        const float4 s4 = scl[(gt & 1) * kTile + row];
        const float sj[4] = {s4.x, s4.y, s4.z, s4.w};
        const int kpos = it.k0 + t * kTile + row;
        bool rv = kpos < it.k0 + it.n;
        if (kSparse) rv = rv && vrow[(gt & 1) * kTile + row] != 0;
        float s[NQ];
        {
          const uint32_t sb = tl + C::kS;
#pragma unroll
          for (int c = 0; c < NQ; ++c) s[c] = 0.f;
          constexpr int kSB = 2;     // S tiles per TMEM round trip (registers)
#pragma unroll
          for (int j = 0; j < 4; j += kSB) {
            float hl[32 * kSB];
            tmem_ld_n<32 * kSB>(sb + 32 * j, hl);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < kSB; ++u)
#pragma unroll
              for (int c = 0; c < NQ; ++c) s[c] = fmaf(sj[j + u], hl[32 * u + c] + hl[32 * u + 16 + c], s[c]);
          }
          float sr[16];
          tmem_ld16(sb + 128, sr);
          tmem_ld_wait();
          // all of S is in this warp's registers: release its lanes of the buffer to the next
          // QK now, ahead of the combine and the vote (one arrival per softmax warp)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free);
#pragma unroll
          for (int c = 0; c < NQ; ++c) s[c] = rv ? p.sig2 * fmaf(colf[c], s[c], sr[c]) : -CUDART_INF_F;
        }
        if (stid == 0) TL(3, 4);
        if (!kSparse) {
          const int dq = kpos - it.L + p.q_len;
          if (rv && dq > 0) {
#pragma unroll
            for (int c = 0; c < NQ; ++c)
              if ((cgb + c) / p.H < dq) s[c] = -CUDART_INF_F;
          }
        }
        bool need = false;
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
          const float mr = mref[c];
          need |= (s[c] > mr + kTau) | ((mr == -CUDART_INF_F) & (s[c] > -CUDART_INF_F));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) need |= rv && (sj[j] * rj[j] > 1.f || rj[j] == 0.f);
        tc_fence_before();
        const bool rare = named_bar_or(1, NT, need || !w);
        if (stid == 0) TL(3, rare ? 6 : 5);
        bool pv_waited = false;
        if (rare) {
          ok = named_bar_and(1, NT, w);
          if (!ok) break;
          float* rb = red_m + (gt & 1) * NQ * 4;
          {
            float v[NQ];
#pragma unroll
            for (int c = 0; c < NQ; ++c) v[c] = s[c];
            const float wm = warp_col_reduce<NQ, true>(v, lane);
            if (lane < 16) rb[lane * 4 + quad] = wm;
            float sm[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              sm[j] = rv ? sj[j] : 0.f;
#pragma unroll
              for (int o = 16; o >= 1; o >>= 1) sm[j] = fmaxf(sm[j], __shfl_xor_sync(0xFFFFFFFFu, sm[j], o));
            }
            if (lane == 0) *reinterpret_cast<float4*>(red_s + quad * 4) = make_float4(sm[0], sm[1], sm[2], sm[3]);
          }
          named_bar_sync(1, NT);
          float mt_l;
          {
            const float4 q4 = reinterpret_cast<const float4*>(rb)[lane % NQ];
            mt_l = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
          }
          bool resc;
          {
            bool moved = false;
            if (lane < NQ) {      // lane c: column c (mt_l holds column lane % NQ)
              const float mo = mref[lane];
              const float mn = fmaxf(mo, mt_l);
              alph[lane] = (mo == -CUDART_INF_F) ? 0.f : ex2(mo - mn);
              moved = (mn != mo);
              mref[lane] = mn;
            }
            resc = __any_sync(0xFFFFFFFFu, moved);
            __syncwarp();
          }
#pragma unroll
          for (int c = 0; c < NQ; ++c) l_part[c] *= alph[c];
          // value-tile references: r_j = 2^-ceil(log2 max s_j) once a larger scale shows up
          {
            bool moved = false;
            if (lane < 4) {       // lane j: value tile j
              const int j = lane;
              float mx = 0.f;
#pragma unroll
              for (int wq = 0; wq < 4; ++wq) mx = fmaxf(mx, red_s[wq * 4 + j]);
              const float ro = rj[j];
              float ra = 1.f;
              if (mx > 0.f && (ro == 0.f || mx * ro > 1.f)) {
                const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127;
                int e = -(ex + ((__float_as_uint(mx) & 0x7FFFFFu) ? 1 : 0));   // 2^e * mx <= 1
                e = max(min(e, 126), -126);
                const float rn = pow2i(e);
                ra = (ro == 0.f) ? 0.f : rn / ro;
                moved = (ro != 0.f);
                rj[j] = rn;
              }
              ratio[j] = ra;
            }
            resc |= __any_sync(0xFFFFFFFFu, moved);
            __syncwarp();
          }
          if (t > 0) {
            w = warp_wait(&pv_done[(gt - 1) & 1], static_cast<uint32_t>((gt - 1) >> 1) & 1u, abort_flag);
            tc_fence_after();
            pv_waited = true;
            if (w && resc) {
#pragma unroll 1
              for (int jq = 0; jq < 4 * (64 / kOB); ++jq) {     // value tile j: four terms x 16 columns
                const int j = jq / (64 / kOB);
                float o[kOB];
                tmem_ld_n<kOB>(tl + C::kTmemO + kOB * jq, o);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < kOB; ++c) o[c] *= alph[c % 16] * ratio[j];
                tmem_st_n<kOB>(tl + C::kTmemO + kOB * jq, o);
              }
              tmem_st_wait();
            }
          }
        }
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
          const float mr = mref[c];
          const float mu = (mr == -CUDART_INF_F) ? 0.f : mr;
          s[c] = ex2(s[c] - mu + kPExp);
          l_part[c] += s[c];
        }
        if (t > 0 && !pv_waited) {
          w = warp_wait(&pv_done[(gt - 1) & 1], static_cast<uint32_t>((gt - 1) >> 1) & 1u, abort_flag);
          tc_fence_after();
        }
        if (stid == 0) TL(3, 7);
        // P_j = p s_j r_j as four e5m2 terms (4 x 16 columns), 8 keys x 16 B core matrices.
        // The first term is P_j rounded to nearest e5m2 from fp32; the rest (exact in fp32, at
        // most 2^-3 of P_j) is rounded once to f16 and split into three more terms: e5m2 is the
        // upper byte of an f16 (same sign, exponent bias and subnormals), so the next two keep
        // the upper byte of what is left (an exact f16 subtraction, which keeps the sign) and
        // the last rounds it to nearest even.  The four carry P_j to about 2^-12 relative.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float f = rv ? sj[j] * rj[j] : 0.f;
          uint8_t* pj = ps + j * (kTile * 64) + (row >> 3) * 512 + (row & 7) * 16;
          uint32_t a[8], w0[4];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float x0 = s[2 * u] * f, x1 = s[2 * u + 1] * f;
            const uint32_t e = e5m2x2_rn(x0, x1);         // column 2u in the low byte
            const float2 t = e5m2x2_to_float2(e);
            const __half2 h = __floats2half2_rn(x0 - t.x, x1 - t.y);
            a[u] = *reinterpret_cast<const uint32_t*>(&h);
            w0[u >> 1] = (u & 1) ? (w0[u >> 1] | (e << 16)) : e;
          }
          *reinterpret_cast<uint4*>(pj) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
#pragma unroll
          for (int term = 1; term < 4; ++term) {
            uint32_t wv[4];
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
              uint32_t t0, t1;
              if (term < 3) {
                t0 = a[u] & 0xFF00FF00u;
                t1 = a[u + 1] & 0xFF00FF00u;
                const __half2 r0 = __hsub2(*reinterpret_cast<const __half2*>(&a[u]), *reinterpret_cast<const __half2*>(&t0));
                const __half2 r1 = __hsub2(*reinterpret_cast<const __half2*>(&a[u + 1]), *reinterpret_cast<const __half2*>(&t1));
                a[u] = *reinterpret_cast<const uint32_t*>(&r0);
                a[u + 1] = *reinterpret_cast<const uint32_t*>(&r1);
              } else {
                t0 = a[u] + 0x007F007Fu + ((a[u] >> 8) & 0x00010001u);
                t1 = a[u + 1] + 0x007F007Fu + ((a[u + 1] >> 8) & 0x00010001u);
              }
              wv[u >> 1] = __byte_perm(t0, t1, 0x7531);
            }
            *reinterpret_cast<uint4*>(pj + 128 * term) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
          // rows past the item or masked: their codes never reach PV (stale slot contents);
          // the gather warps already store zeros for them
          if (!kSparse && !rv) {
            uint4* dst = reinterpret_cast<uint4*>(ring + ((gt & 1) * NB + j) * kSlotBytes + row * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          }
          // P_j of this warp's 32 keys is in place: PV of value tile j may start (the O
          // rescale above has completed; a warp whose PV wait failed does not arrive, and the
          // issuer's bounded wait then ends on the abort word)
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && w) mbar_arrive(&p_full[j]);
        }
        if (stid == 0) TL(3, 8);
        ok = named_bar_and(1, NT, w);
        if (!ok) break;
      }
      if (!ok) break;
      // The next item's query, ahead of this item's epilogue, when that item is already posted:
      // QK of this item's last tile is done (its S was read), so the query buffer and the
      // column factors are free, and the next item's QK then overlaps this epilogue (its PV
      // still waits for its P, written after the epilogue has read O out).
      {
        const int kn = nit % kItemDepth;
        const bool posted = mbar_test_wait(&item_full[kn], static_cast<uint32_t>(nit / kItemDepth) & 1u);
        if (named_bar_and(1, NT, posted)) {
          const WorkItem nx = items[kn];
          if (nx.b >= 0 && nx.ntiles > 0) {
            prep_query(nx);
            q_ready = true;
          }
        }
      }
      // ---- epilogue
      w = true;
      if (it.ntiles > 0) {
        w = warp_wait(&pv_done[(g + it.ntiles - 1) & 1], static_cast<uint32_t>((g + it.ntiles - 1) >> 1) & 1u,
                      abort_flag);
        tc_fence_after();
      }
      g += it.ntiles;
      {
        const float lw = warp_col_reduce<NQ, false>(l_part, lane);
        if (lane < 16) red_l[lane * 4 + quad] = lw;
      }
      ok = named_bar_and(1, NT, w);
      if (!ok) break;
      const int cl = lane % NQ;
      float inv_l, lse_l;
      {
        const float4 q4 = reinterpret_cast<const float4*>(red_l)[cl];
        const float l = (q4.x + q4.y) + (q4.z + q4.w);
        const float m_l = mref[cl];
        const bool live = l > 0.f;
        inv_l = live ? __fdividef(1.f, l) : 0.f;
        lse_l = live ? (m_l + __log2f(l) - kPExp) * 0.69314718055994531f : -CUDART_INF_F;
      }
      float inv[NQ];
#pragma unroll
      for (int c = 0; c < NQ; ++c) inv[c] = __shfl_sync(0xFFFFFFFFu, inv_l, c);
      const bool final_out = !p.partial;
      const int64_t flat0 = static_cast<int64_t>(it.b) * p.q_len * p.H + cgb;
      const int ncol = min(NQ, p.cols - cgb);
      const int qi0 = cgb / p.H, h0 = cgb % p.H;
      const int64_t o_wrap = p.o_s0b - static_cast<int64_t>(p.H) * p.o_s1b;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        float o[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) o[c] = 0.f;
        if (it.ntiles > 0) {
          float ot[64];
          tmem_ld_n<64>(tl + C::kTmemO + 64 * j, ot);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) o[c] = (ot[c] + ot[16 + c]) + (ot[32 + c] + ot[48 + c]);
        }
        const float ur = (rj[j] > 0.f) ? 1.f / rj[j] : 0.f;     // exact: a power of two
        const int d = 128 * j + row;
        if (final_out && (kSparse || p.q_len == 1)) {
          // One query token per row (always so for the sparse rows): the group's columns are
          // heads cgb .. cgb + ncol - 1 of one token and never wrap.
          uint8_t* ptr = p.out + static_cast<int64_t>(it.b) * p.o_s0b + static_cast<int64_t>(cgb) * p.o_s1b + 2 * d;
#pragma unroll
          for (int c = 0; c < NQ; ++c) {
            if (c < ncol) *reinterpret_cast<__nv_bfloat16*>(ptr) = __float2bfloat16_rn(o[c] * ur * inv[c]);
            ptr += p.o_s1b;
          }
        } else if (final_out) {
          // Running pointer over (token, head): column c + 1 is the next head, or head 0 of the
          // next token after head H - 1 (no per-store index multiply).
          uint8_t* ptr = p.out + (static_cast<int64_t>(it.b) * p.q_len + qi0) * p.o_s0b +
                         static_cast<int64_t>(h0) * p.o_s1b + 2 * d;
          int h = h0;
#pragma unroll
          for (int c = 0; c < NQ; ++c) {
            if (c < ncol) *reinterpret_cast<__nv_bfloat16*>(ptr) = __float2bfloat16_rn(o[c] * ur * inv[c]);
            ptr += p.o_s1b;
            if (++h == p.H) {
              h = 0;
              ptr += o_wrap;
            }
          }
        } else {
          float* dst = p.part_o + ((static_cast<int64_t>(it.s) * p.n_rows * p.H + flat0) * kLora + d);
#pragma unroll
          for (int c = 0; c < NQ; ++c)
            if (c < ncol) dst[static_cast<int64_t>(c) * kLora] = o[c] * ur * inv[c];
        }
      }
      if (row < 16 && cl < ncol) {
        if (final_out) {
          if (p.lse) p.lse[flat0 + cl] = lse_l;
        } else {
          p.part_lse[static_cast<int64_t>(it.s) * p.n_rows * p.H + flat0 + cl] = lse_l;
        }
      }
      tc_fence_before();
      named_bar_sync(1, NT);
      if (stid == 0) mbar_arrive(&item_empty[k]);
    }
  } else if (warp == C::kPvWarp) {
    // ------------------------------------------------------------------ PV issuer
    // A second MMA-issuing thread: PV(t) goes to the tensor cores as soon as P(t) is written,
    // in parallel with the QK of the next tile (a commit tracks the issuing thread's MMAs).
    if (lane == 0) {
      const uint64_t dV0 = smem_desc(smem_u32(ring), kSlotBytes, 1024, kSwizzle128B);
      const uint64_t dP0 = smem_desc(smem_u32(ps), 512, 128, kSwizzleNone);
      constexpr uint32_t kIdPv = idesc_e4m3(128, 64, 1, 1) | (1u << 10);   // B (weights) in e5m2
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
          TL(1, 3);
          for (int j = 0; j < 4 && ok; ++j) {
            ok = mbar_wait(&p_full[j], static_cast<uint32_t>(gt) & 1u, abort_flag);
            tc_fence_after();
            if (ok) ds_issue_pv_block<NB>(tmem + C::kTmemO, dV0, dP0, kIdPv, gt, j, t == 0);
          }
          if (!ok) break;
          mma_commit(&pv_done[gt & 1]);
          // cluster: this CTA's share of "tile gt's slots are free", in every CTA
          if (kCl > 1) mma_commit_mc(&ring_free[gt & 1], kMask);
          TL(1, 4);
        }
        g += it.ntiles;
      }
      mma_commit(fin_pv);
      volatile int no_abort[2] = {0, 0};
      mbar_wait(fin_pv, 0, no_abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ gather (sparse)
    // Gather warp w (0..7) loads records 16 w .. 16 w + 15 of the tile; a record is 41 16-byte
    // chunks (0..31 codes, 32 scales, 33..40 k_pe).  Loads are coalesced per record: load
    // i < 16 brings the 32 code chunks of record 16 w + i (lane l: chunk l), and loads 16..20
    // bring the 9 other chunks of all 16 records (lane l of load 16 + u: flat chunk
    // f = 32 u + l < 144, record f / 9, chunk 32 + f % 9).  The tile waits in registers while
    // its ring slots drain.
    const int gw = warp - 6, rbase = 16 * gw;
    uint32_t errbits = 0;
    int nit = 0, g = 0;
    bool ok = true;
    while (ok) {
      const int k = nit % kItemDepth;
      if (!warp_wait(&item_full[k], (nit / kItemDepth) & 1, abort_flag)) break;
      const WorkItem it = items[k];
      ++nit;
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[k]);
      if (it.b < 0) break;
      // lane l < 16: the index of record rbase + l of tile tt, loaded one tile ahead (its
      // latency then hides behind this tile's wait and stores) and checked when used
      auto raw_index = [&](int tt) -> int {
        const int e = tt * kTile + rbase + lane;
        return (lane < 16 && tt < it.ntiles && e < it.n) ? p.indices[it.k0 + e] : -1;
      };
      int raw_nx = raw_index(0);
      for (int t = 0; t < it.ntiles && ok; ++t) {
        const int gt = g + t;
        // lane l < 16: record rbase + l of the tile (-1: past the row, masked or bad)
        int idx = -1;
        if (lane < 16 && t * kTile + rbase + lane < it.n) {
          idx = raw_nx;
          if (idx < 0 || idx >= p.num_records) {
            if (idx >= p.num_records || !p.has_invalid) errbits |= 1u;
            idx = -1;
          }
        }
        if (lane == 0) TL(4 + gw, 1);
        uint4 v[21];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int ri = __shfl_sync(0xFFFFFFFFu, idx, i);
          v[i] = (ri >= 0) ? *reinterpret_cast<const uint4*>(p.records + static_cast<int64_t>(ri) * p.rec_stride + 16 * lane)
                           : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 5; ++u) {
          const int f = 32 * u + lane, rr = f / 9, c = 32 + f - 9 * rr;
          const int ri = __shfl_sync(0xFFFFFFFFu, idx, rr & 15);
          v[16 + u] = (f < 144 && ri >= 0)
                          ? *reinterpret_cast<const uint4*>(p.records + static_cast<int64_t>(ri) * p.rec_stride + 16 * c)
                          : make_uint4(0, 0, 0, 0);
        }
        raw_nx = raw_index(t + 1);
        // tile gt reuses the slots of tile gt - 2
        if (gt >= 2 && !warp_wait(&pv_done[gt & 1], static_cast<uint32_t>((gt - 2) >> 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) TL(4 + gw, 2);
        {
          uint8_t* codes = ring + ((gt & 1) * NB + (lane >> 3)) * kSlotBytes;
#pragma unroll
          for (int i = 0; i < 16; ++i) *reinterpret_cast<uint4*>(codes + sw128(rbase + i, lane & 7)) = v[i];
        }
#pragma unroll
        for (int u = 0; u < 5; ++u) {
          const int f = 32 * u + lane, rr = f / 9, c = 32 + f - 9 * rr;
          if (f < 144) {
            const int r = rbase + rr;
            if (c == 32)
              *reinterpret_cast<uint4*>(scl + (gt & 1) * kTile + r) = v[16 + u];
            else
              *reinterpret_cast<uint4*>(ring + ((gt & 1) * NB + 4) * kSlotBytes + sw128(r, c - 33)) = v[16 + u];
          }
        }
        if (lane < 16) vrow[(gt & 1) * kTile + rbase + lane] = (idx >= 0) ? 1 : 0;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[(gt & 1) * NB]);     // the tile's one full barrier
        if (lane == 0) TL(4 + gw, 3);
      }
      g += it.ntiles;
    }
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (lane == 0 && errbits) set_device_error(p.err, errbits);
  }

  tc_fence_before();
  __syncthreads();
  if (kCl > 1) {
    // cluster: every producer has stopped issuing; wait (bounded) until every copy that any
    // of them issued into this CTA's ring has landed, so that no copy targets it once it exits.
    // A position that one producer never issued (after an abort) keeps its phase open: the
    // wait then runs to its limit, by which time the other copies of that position have landed.
    cluster_sync();
    if (tid == 0) {
      int64_t hi = 0;
      for (int r = 0; r < kCl; ++r) hi = max(hi, cl_pos[r]);
      const int64_t first = hi > R ? hi - R : 0;
      volatile int drain[2] = {0, 0};
      for (int64_t q = first; q < hi; ++q)
        if (!mbar_wait(&full[q % R], static_cast<uint32_t>(q / R) & 1u, drain)) break;
    }
    __syncthreads();
  }
  if (tid == 0 && *abort_flag == 2) set_device_error(p.err, 16u);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace mla
