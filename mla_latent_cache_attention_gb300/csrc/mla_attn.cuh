// mla_attn.cuh -- MLA attention over the 576-wide latent cache on tcgen05 tensor cores.
//
// One kernel template serves both key sources of the path:
//   * sparse (CSR key lists over fp8_ds_mla records): "vllm.models.kimi_k3.amd.ops.
//     flydsl_sparse_mla", flydsl_sparse_mla_fp8ds_fwd;
//   * paged decode / spec-verify (bf16, plain fp8, fp8_ds_mla caches, split-K over the key
//     sequence): "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.prepared",
//     PreparedMla.stock_core and trtllm_decode.
//
// Work item = (query row, group of 16 heads, key split).  All 16 heads of a row share every
// key (MQA), so the products run "swap-AB" on the tensor core: M = 128 keys (TMEM lanes),
// N = 16 heads, K = the 576 (QK) or 128-key (PV) contraction.
//
//   QK:  S^T[key, h]  = K_tile[128 x 576] . Q^T           (A: key tile, K-major SW128)
//   PV:  O^T[d, h]   += V^T[128 d x 128 keys] . P^T        (A: the same tile, MN-major)
//
// Exactness of the fp8_ds_mla path: the 512 NoPE codes are converted to f16 exactly (no
// scale folded in); QK runs as four separate accumulators, one per 128-wide tile j, plus a
// bf16 one for the rope part, and S = sum_j scale_j[key] * S_j + S_rope is formed in fp32.
// PV folds scale_j into P (four P matrices, one per output tile j).  Plain fp8 converts all
// 576 codes to f16 exactly (q too); bf16 uses the cache bytes as they are.
//
// CTA = 10 warps: warp 0 gathers entries with 1-D bulk copies into a staging ring (and
// prefetches two tiles ahead into L2), warp 1 issues the MMAs (one thread) and owns TMEM,
// warps 6..9 convert staged entries into the swizzled operand tile (one thread per entry),
// warps 2..5 run the online softmax (one thread per key lane) and the epilogue (one thread
// per output column d).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "mla_ptx.cuh"

namespace mla {

enum : int { kBF16 = 0, kFP8 = 1, kDS = 2 };

#ifdef MLA_TIMELINE
// Debug timeline (never in the product build): per CTA (first 4) and role, a log of
// (event id, %globaltimer) pairs.  Store-only: the marking thread counts in a register.
constexpr int kTlCtas = 4, kTlRoles = 12, kTlEvents = 512;
__device__ unsigned long long g_tl[kTlCtas][kTlRoles][kTlEvents][2];
__device__ int g_tl_n[kTlCtas][kTlRoles];
__device__ __forceinline__ void tl_mark(int role, int ev, int& n) {
  if (blockIdx.x < kTlCtas && n < kTlEvents) {
    g_tl[blockIdx.x][role][n][0] = ev;
    g_tl[blockIdx.x][role][n][1] = globaltimer();
    ++n;
    g_tl_n[blockIdx.x][role] = n;
  }
}
#define TL(role, ev) tl_mark(role, ev, tl_n)
#define TL_DECL int tl_n = 0
#else
#define TL(role, ev) ((void)0)
#define TL_DECL ((void)0)
#endif


constexpr int kTile = 128;               // keys per tile (MMA M, TMEM lanes)
constexpr int kRows = 16;                // heads per CTA (MMA N)
constexpr int kEntry = 576, kLora = 512;
constexpr int kBlk = 9;                  // 64-wide blocks of d in 576
constexpr int kBlkBytes = kTile * 128;   // one SW128 block of the key tile: 128 rows x 128 B
constexpr int kQBlkBytes = kRows * 128;  // one SW128 block of the query tile
constexpr int kThreads = 320;            // 10 warps, see the role map below
constexpr int kTmemCols = 256;
constexpr int kOCol = 128;               // TMEM column of the O^T accumulators
constexpr int kSmemLimit = 232448;       // opt-in shared memory per block on sm_100-class parts

// Per-format staging: entries are gathered with one bulk copy each into a staging piece of
// kPiece entries at a pitch of kRecPad bytes (an odd number of 16-byte units, so that one
// thread per entry reads shared memory without bank conflicts).
template <int F> struct Fmt;
template <> struct Fmt<kBF16> {
  static constexpr int kRec = 1152, kRecPad = 1168, kPiece = 16, kStages = 3, kNP = 1;
};
template <> struct Fmt<kFP8> {
  static constexpr int kRec = 576, kRecPad = 592, kPiece = 32, kStages = 2, kNP = 1;
};
template <> struct Fmt<kDS> {
  static constexpr int kRec = 656, kRecPad = 656, kPiece = 32, kStages = 2, kNP = 4;
};

template <int F> struct Smem {
  static constexpr int kKV = 0;
  static constexpr int kQ = kKV + kBlk * kBlkBytes;               // 147456
  static constexpr int kP = kQ + kBlk * kQBlkBytes;                // +18432
  static constexpr int kStage = kP + Fmt<F>::kNP * 4096;
  static constexpr int kStageBytes = Fmt<F>::kPiece * Fmt<F>::kRecPad;
  static constexpr int kScale = kStage + Fmt<F>::kStages * kStageBytes;   // [128][4] fp32
  static constexpr int kValid = kScale + kTile * 16;               // [128] u8
  static constexpr int kRed = kValid + kTile;                      // [2][4][16] + [4][16] fp32
  static constexpr int kAddr = kRed + 3 * 4 * 16 * 4;              // [2][128] entry addresses
  static constexpr int kBar = kAddr + 2 * kTile * 8;               // mbarriers (8-byte aligned)
  static constexpr int kNumBars = 2 * Fmt<F>::kStages + 5;
  static constexpr int kMisc = kBar + kNumBars * 8;                // meta[kStages], tmem addr, abort
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kAlloc = kTotal + 1024;                     // slack for 1024-B alignment
  static_assert(kAlloc <= kSmemLimit, "shared memory budget");
  static_assert(kStage % 16 == 0 && kStageBytes % 16 == 0, "bulk copy alignment");
};

struct AttnParams {
  // queries: [n_rows, H, 576] (bf16, or e4m3 bytes for the plain fp8 cache)
  const uint8_t* q;
  int64_t q_s0b, q_s1b;   // byte strides
  int H, n_hgroups;
  // sparse key source
  const uint8_t* records;
  int64_t rec_stride, num_records;
  const int32_t* indptr;
  const int32_t* indices;
  int has_invalid;
  // paged key source
  const uint8_t* cache;
  int64_t num_blocks, block_stride, entry_stride;
  int block_size;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;
  int q_len;
  int64_t chunk;          // keys per split (multiple of kTile)
  int n_splits;
  int tma_rows;           // TMA page kernel: rows per box (divides 128)
  // items
  int n_rows, n_items;
  // scales
  float sig2;             // logit scale times log2(e)
  float out_scale;
  // outputs
  uint8_t* out;           // bf16 [n_rows, H, >=512] (final) -- used when n_splits == 1
  int64_t o_s0b, o_s1b;
  float* lse;             // [n_rows, H] or null
  float* part_o;          // [n_splits][n_rows][H][512] fp32 -- used when n_splits > 1
  float* part_lse;        // [n_splits][n_rows][H]
  uint32_t* err;
};

struct ItemInfo {
  int row, hg, split;
  int64_t k0;   // first entry index (sparse) / first key position (paged)
  int64_t n;    // keys (entries) in the item
};

template <bool kSparse>
__device__ __forceinline__ ItemInfo decode_item(const AttnParams& p, int item) {
  ItemInfo it;
  it.hg = item % p.n_hgroups;
  int rs = item / p.n_hgroups;
  it.split = rs % p.n_splits;
  it.row = rs / p.n_splits;
  if (kSparse) {
    int64_t b = p.indptr[it.row], e = p.indptr[it.row + 1];
    it.k0 = b;
    it.n = e > b ? e - b : 0;
  } else {
    int b = it.row / p.q_len, i = it.row % p.q_len;
    int64_t L = p.seq_lens[b];
    int64_t vis = L - p.q_len + i + 1;
    if (vis < 0) vis = 0;
    int64_t s0 = static_cast<int64_t>(it.split) * p.chunk;
    int64_t s1 = (it.split == p.n_splits - 1) ? vis : min(vis, s0 + p.chunk);
    it.k0 = s0;
    it.n = s1 > s0 ? s1 - s0 : 0;
  }
  return it;
}

// Address of key k of an item, or nullptr when the key is masked / out of range.
template <bool kSparse>
__device__ __forceinline__ const uint8_t* key_entry(const AttnParams& p, const ItemInfo& it,
                                                    int64_t k, uint32_t& errbits) {
  if (kSparse) {
    int32_t idx = p.indices[it.k0 + k];
    if (idx < 0) {
      if (!p.has_invalid) errbits |= 1u;
      return nullptr;
    }
    if (idx >= p.num_records) {
      errbits |= 1u;
      return nullptr;
    }
    return p.records + static_cast<int64_t>(idx) * p.rec_stride;
  } else {
    int64_t pos = it.k0 + k;
    int b = it.row / p.q_len;
    int64_t blk = p.block_table[static_cast<int64_t>(b) * p.bt_stride + pos / p.block_size];
    if (blk < 0 || blk >= p.num_blocks) {
      errbits |= 2u;
      return nullptr;
    }
    return p.cache + blk * p.block_stride + (pos % p.block_size) * p.entry_stride;
  }
}

// Keys in tile t of an item with n keys.
__device__ __forceinline__ int tile_keys(int64_t n, int t) {
  const int64_t r = n - static_cast<int64_t>(t) * kTile;
  return static_cast<int>(r < kTile ? r : kTile);
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes & 0xFFFFu),
                                             __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 raw) {
  uint4 o;
  o.x = e4m3x2_to_f16x2(raw.x);
  o.y = e4m3x2_to_f16x2(raw.x >> 16);
  o.z = e4m3x2_to_f16x2(raw.y);
  o.w = e4m3x2_to_f16x2(raw.y >> 16);
  return o;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v);
  float2 f = __bfloat1622float2(b);
  __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Query chunk (8 values = 16 bytes) of block b (0..8), chunk c (0..7), in the operand type
// the key tile uses for that block: f16 for the e4m3-sourced blocks, bf16 otherwise.
template <int F>
__device__ __forceinline__ uint4 query_chunk(const uint8_t* qrow, int b, int c) {
  if (F == kFP8) {
    return e4m3x8_to_f16x8(*reinterpret_cast<const uint2*>(qrow + 64 * b + 8 * c));
  }
  uint4 v = *reinterpret_cast<const uint4*>(qrow + 128 * b + 16 * c);
  if (F == kDS && b < 8) {
    v.x = bf16x2_to_f16x2(v.x);
    v.y = bf16x2_to_f16x2(v.y);
    v.z = bf16x2_to_f16x2(v.z);
    v.w = bf16x2_to_f16x2(v.w);
  }
  return v;
}

__device__ __forceinline__ uint32_t sw128(int row, int c) {
  return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool as_bf16) {
  if (as_bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// L2 prefetch of an entry, one instruction per 128-byte line (the bulk-copy engine is kept
// for the copies themselves).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  const uint8_t* c = static_cast<const uint8_t*>(p);
  for (uint32_t off = 0; off < bytes; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

// One converter thread turns 64 consecutive e4m3 bytes of its staged entry into one 64-wide
// f16 block row of the key tile (8 swizzled 16-byte chunks); `sw` holds the row's swizzled
// chunk offsets.  All loads are issued before any store.
__device__ __forceinline__ void cvt_block_e4m3(const uint8_t* src, uint8_t* dst_row, const uint32_t (&sw)[8],
                                               bool valid) {
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) raw[i] = valid ? *reinterpret_cast<const uint4*>(src + 16 * i) : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 lo = e4m3x8_to_f16x8(make_uint2(raw[i].x, raw[i].y));
    const uint4 hi = e4m3x8_to_f16x8(make_uint2(raw[i].z, raw[i].w));
    *reinterpret_cast<uint4*>(dst_row + sw[2 * i]) = lo;
    *reinterpret_cast<uint4*>(dst_row + sw[2 * i + 1]) = hi;
  }
}

// Same for 64 16-bit values copied as they are.
__device__ __forceinline__ void copy_block_16b(const uint8_t* src, uint8_t* dst_row, const uint32_t (&sw)[8],
                                               bool valid) {
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = valid ? *reinterpret_cast<const uint4*>(src + 16 * i) : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(dst_row + sw[i]) = v[i];
}

// Converter warp cw (0..3) writes blocks 2cw and 2cw+1 of key-tile row `row` from the staged
// entry `rec`; warp 3 also writes block 8 (d 512..575) and, for fp8_ds_mla, the tile scales.
template <int F>
__device__ __forceinline__ void convert_row(const uint8_t* rec, bool valid, uint8_t* kv, int row, int cw,
                                            float* scales) {
  uint32_t sw[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) sw[c] = static_cast<uint32_t>(((c ^ (row & 7)) << 4));
  uint8_t* base = kv + row * 128;
#pragma unroll
  for (int bb = 0; bb < 2; ++bb) {
    const int b = 2 * cw + bb;
    if (F == kBF16)
      copy_block_16b(rec + 128 * b, base + b * kBlkBytes, sw, valid);
    else
      cvt_block_e4m3(rec + 64 * b, base + b * kBlkBytes, sw, valid);
  }
  if (cw == 3) {
    if (F == kBF16)
      copy_block_16b(rec + 1024, base + 8 * kBlkBytes, sw, valid);
    else if (F == kFP8)
      cvt_block_e4m3(rec + 512, base + 8 * kBlkBytes, sw, valid);
    else
      copy_block_16b(rec + 528, base + 8 * kBlkBytes, sw, valid);
    if (F == kDS) {
      float4 sc = valid ? *reinterpret_cast<const float4*>(rec + 512) : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(scales + row * 4) = sc;
    }
  }
}

// Warp-wide max (or sum) of 16 per-thread values, one per head: a halving butterfly leaves
// the result for head (lane >> 1) & 15 in every lane (16 shuffles instead of 80).
template <bool kMax>
__device__ __forceinline__ float butterfly16(const float (&v)[16], int lane) {
  float a[8], b4[4], c2[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = u16 ? v[i] : v[i + 8];
    const float keep = u16 ? v[i + 8] : v[i];
    const float got = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    a[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = u8 ? a[i] : a[i + 4];
    const float keep = u8 ? a[i + 4] : a[i];
    const float got = __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    b4[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u4 ? b4[i] : b4[i + 2];
    const float keep = u4 ? b4[i + 2] : b4[i];
    const float got = __shfl_xor_sync(0xFFFFFFFFu, send, 4);
    c2[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
  const float send = u2 ? c2[0] : c2[1];
  const float keep = u2 ? c2[1] : c2[0];
  float r = keep;
  {
    const float got = __shfl_xor_sync(0xFFFFFFFFu, send, 2);
    r = kMax ? fmaxf(keep, got) : keep + got;
  }
  const float got = __shfl_xor_sync(0xFFFFFFFFu, r, 1);
  return kMax ? fmaxf(r, got) : r + got;
}
// The head whose reduction butterfly16 leaves in `lane`.
__device__ __forceinline__ int butterfly16_head(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// ------------------------------------------------------------------------------------------
// The kernel.  Warp roles:
//   0      producer: per-entry 1-D bulk copies into the staging ring; entry addresses and an L2
//          prefetch one tile ahead;
//   1      MMA issuer (one thread) and TMEM owner;
//   2..5   softmax + epilogue: thread = TMEM lane = key row of the tile (logits) and output
//          column d (O^T readout);
//   6..9   converters: staged entries -> swizzled f16 / bf16 key tile, thread = entry.
// Every wait is bounded; softmax warps vote at their named barriers so they leave together.
template <int F, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1) mla_attn_kernel(const __grid_constant__ AttnParams p) {
  using FT = Fmt<F>;
  using SM = Smem<F>;
  constexpr int NST = FT::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem + SM::kKV;
  uint8_t* qs = smem + SM::kQ;
  uint8_t* ps = smem + SM::kP;
  uint8_t* stage = smem + SM::kStage;
  float* scales = reinterpret_cast<float*>(smem + SM::kScale);
  uint8_t* valid_row = smem + SM::kValid;
  float* red = reinterpret_cast<float*>(smem + SM::kRed);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + NST;
  uint64_t* tile_full = bars + 2 * NST;
  uint64_t* s_full = tile_full + 1;
  uint64_t* p_full = tile_full + 2;
  uint64_t* o_done = tile_full + 3;
  uint64_t* mma_final = tile_full + 4;
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + SM::kMisc);
  uint32_t* tmem_slot = meta + NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(meta + NST + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  TL_DECL;

  // the split-K merge may be scheduled now; it waits for this grid to complete
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);      // one arrival per converter warp
    }
    mbar_init(tile_full, 4);        // one arrival per converter warp
    mbar_init(s_full, 1);
    mbar_init(p_full, 1);
    mbar_init(o_done, 1);
    mbar_init(mma_final, 1);
    *abort_flag = 0;
    abort_flag[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
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
    // Entry addresses of a tile are resolved one tile ahead (four independent index / block-
    // table loads per lane, in flight while the current tile's copies are issued) into a
    // two-slot ring in shared memory, and prefetched into L2 from there.
    const uint8_t** addr_ring = reinterpret_cast<const uint8_t**>(smem + SM::kAddr);
    int st = 0;
    uint32_t eph = 0;
    uint32_t errbits = 0;
    bool armed[NST] = {};
    uint32_t armed_par[NST] = {};
    bool ok = true;
    struct Cursor {
      int item, t, ntiles;
      ItemInfo it;
    };
    auto first_from = [&](int item) {
      Cursor c{item, 0, 0, ItemInfo{}};
      for (; c.item < p.n_items; c.item += gridDim.x) {
        c.it = decode_item<kSparse>(p, c.item);
        c.ntiles = static_cast<int>((c.it.n + kTile - 1) / kTile);
        if (c.ntiles > 0) return c;
      }
      return c;
    };
    auto advance = [&](const Cursor& c) {
      if (c.t + 1 < c.ntiles) {
        Cursor n = c;
        n.t += 1;
        return n;
      }
      return first_from(c.item + gridDim.x);
    };
    auto tile_addrs = [&](const Cursor& c, const uint8_t* (&a)[4]) {
      const int nk = tile_keys(c.it.n, c.t);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = lane + 32 * i;
        a[i] = (k < nk) ? key_entry<kSparse>(p, c.it, static_cast<int64_t>(c.t) * kTile + k, errbits) : nullptr;
      }
    };
    auto publish = [&](const uint8_t* (&a)[4], int slot_) {
      const uint8_t** ring = addr_ring + slot_ * kTile;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ring[lane + 32 * i] = a[i];
        if (a[i]) prefetch_l2(a[i], FT::kRec);
      }
    };
    Cursor cur = first_from(blockIdx.x);
    int slot = 0;
    if (cur.item < p.n_items) {
      const uint8_t* a[4];
      tile_addrs(cur, a);
      publish(a, 0);
      __syncwarp();
    }
    while (ok && cur.item < p.n_items) {
      const Cursor nxt = advance(cur);
      const uint8_t* an[4] = {nullptr, nullptr, nullptr, nullptr};
      if (nxt.item < p.n_items) tile_addrs(nxt, an);
      const int nk = tile_keys(cur.it.n, cur.t);
      const int npieces = (nk + FT::kPiece - 1) / FT::kPiece;
      const uint8_t* const* ring = addr_ring + slot * kTile;
      for (int pc = 0; pc < npieces; ++pc) {
        if (!mbar_wait(&empty[st], eph ^ 1u, abort_flag)) { ok = false; break; }
        const int kin = pc * FT::kPiece + lane;
        const uint8_t* src = (lane < FT::kPiece && kin < nk) ? ring[kin] : nullptr;
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, src != nullptr);
        // entries that sit back to back at the staging pitch (a page of an unpadded cache)
        // arrive with one copy instead of one per entry
        const int cnt = min(FT::kPiece, nk - pc * FT::kPiece);
        const uint8_t* src0 = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xFFFFFFFFu, static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(src)), 0));
        const bool contig = (FT::kRecPad == FT::kRec) && mask == ((cnt >= 32) ? 0xFFFFFFFFu : ((1u << cnt) - 1u)) &&
                            __all_sync(0xFFFFFFFFu, lane >= cnt || src == src0 + static_cast<int64_t>(lane) * FT::kRec);
        if (lane == 0) {
          meta[st] = mask;
          mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(__popc(mask)) * FT::kRec);
          if (contig) bulk_g2s(stage + st * SM::kStageBytes, src0, static_cast<uint32_t>(cnt) * FT::kRec, &full[st]);
        }
        __syncwarp();
        if (!contig && src) bulk_g2s(stage + st * SM::kStageBytes + lane * FT::kRecPad, src, FT::kRec, &full[st]);
        armed[st] = true;
        armed_par[st] = eph;
        if (++st == NST) { st = 0; eph ^= 1u; }
      }
      if (!ok) break;
      slot ^= 1;
      if (nxt.item < p.n_items) publish(an, slot);
      __syncwarp();
      cur = nxt;
    }
    volatile int no_abort[2] = {0, 0};     // never leave bulk copies in flight behind us
    for (int s = 0; s < NST; ++s)
      if (armed[s]) mbar_wait(&full[s], armed_par[s], no_abort);
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (lane == 0 && errbits) set_device_error(p.err, errbits);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t kv_a = smem_u32(kv), q_a = smem_u32(qs), p_a = smem_u32(ps);
      // descriptors differ only in their start-address field (16-byte units; shared addresses
      // stay below 256 KB, so adding to the 14-bit field never carries out of it)
      const uint64_t dK = smem_desc(kv_a, 16, 1024, kSwizzle128B);
      const uint64_t dQ = smem_desc(q_a, 16, 1024, kSwizzle128B);
      const uint64_t dV = smem_desc(kv_a, kBlkBytes, 1024, kSwizzle128B);
      const uint64_t dP = smem_desc(p_a, 256, 128, kSwizzleNone);
      constexpr uint32_t kIdQkNope = idesc_f16(128, kRows, F == kBF16, F == kBF16, 0, 0);
      constexpr uint32_t kIdQkRope = idesc_f16(128, kRows, 1, 1, 0, 0);
      constexpr uint32_t kIdPv = idesc_f16(128, kRows, F == kBF16, F == kBF16, 1, 1);
      uint32_t ph_t = 0, ph_p = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const ItemInfo it = decode_item<kSparse>(p, item);
        const int ntiles = static_cast<int>((it.n + kTile - 1) / kTile);
        for (int t = 0; t < ntiles; ++t) {
          TL(2, 1);
          if (!mbar_wait(tile_full, ph_t, abort_flag)) { ok = false; break; }
          TL(2, 2);
          ph_t ^= 1u;
          tc_fence_after();
          if (F == kDS) {
            for (int j = 0; j < 4; ++j)
              for (int kk = 0; kk < 8; ++kk) {
                const int b = 2 * j + (kk >> 2);
                const uint32_t ko = (kk & 3) * 32;
                mma_f16_ss(tmem + 16 * j, dK + ((b * kBlkBytes + ko) >> 4), dQ + ((b * kQBlkBytes + ko) >> 4),
                           kIdQkNope, kk > 0);
              }
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t ko = kk * 32;
              mma_f16_ss(tmem + 64, dK + ((8 * kBlkBytes + ko) >> 4), dQ + ((8 * kQBlkBytes + ko) >> 4), kIdQkRope,
                         kk > 0);
            }
          } else {
            for (int ks = 0; ks < 36; ++ks) {
              const int b = ks >> 2;
              const uint32_t ko = (ks & 3) * 32;
              mma_f16_ss(tmem, dK + ((b * kBlkBytes + ko) >> 4), dQ + ((b * kQBlkBytes + ko) >> 4), kIdQkNope, ks > 0);
            }
          }
          mma_commit(s_full);
          TL(2, 3);
          if (!mbar_wait(p_full, ph_p, abort_flag)) { ok = false; break; }
          TL(2, 4);
          ph_p ^= 1u;
          tc_fence_after();
          for (int j = 0; j < 4; ++j)
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t a = dV + ((2 * j * kBlkBytes + kk * 2048) >> 4);
              const uint64_t b = dP + (((F == kDS ? j * 4096 : 0) + kk * 512) >> 4);
              mma_f16_ss(tmem + kOCol + 16 * j, a, b, kIdPv, (t > 0 || kk > 0) ? 1u : 0u);
            }
          mma_commit(o_done);
          TL(2, 5);
        }
      }
      mma_commit(mma_final);
      volatile int no_abort[2] = {0, 0};
      mbar_wait(mma_final, 0, no_abort);
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------------ converters
    const int cw = warp - 6;
    const int ct = tid - 192;           // 0..127
    int st = 0;
    uint32_t sph = 0, ph_o = 0;
    bool first = true, ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
      const ItemInfo it = decode_item<kSparse>(p, item);
      const int ntiles = static_cast<int>((it.n + kTile - 1) / kTile);
      const int h0 = it.hg * kRows;
      const int nh = min(kRows, p.H - h0);
      for (int t = 0; t < ntiles && ok; ++t) {
        // the key tile (and at an item start the query tile) is free once the previous PV is done
        if (cw == 0 && lane == 0) TL(1, 1);
        if (!first) {
          if (!mbar_wait(o_done, ph_o, abort_flag)) { ok = false; break; }
          ph_o ^= 1u;
        }
        if (cw == 0 && lane == 0) TL(1, 2);
        first = false;
        if (t == 0) {
          for (int i = ct; i < kRows * 72; i += 128) {
            const int r = i / 72, rem = i % 72, b = rem >> 3, c = rem & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < nh) v = query_chunk<F>(p.q + it.row * p.q_s0b + (h0 + r) * p.q_s1b, b, c);
            *reinterpret_cast<uint4*>(qs + b * kQBlkBytes + sw128(r, c)) = v;
          }
        }
        const int nk = tile_keys(it.n, t);
        const int npieces = (nk + FT::kPiece - 1) / FT::kPiece;
        for (int pc = 0; pc < npieces; ++pc) {
          if (cw == 0 && lane == 0) TL(1, 3);
          if (!mbar_wait(&full[st], sph, abort_flag)) { ok = false; break; }
          if (cw == 0 && lane == 0) TL(1, 4);
          const uint32_t mask = meta[st];
          if (lane < FT::kPiece) {
            const int row = pc * FT::kPiece + lane;
            const bool v = (mask >> lane) & 1u;
            convert_row<F>(stage + st * SM::kStageBytes + lane * FT::kRecPad, v, kv, row, cw, scales);
            if (cw == 3) valid_row[row] = v ? 1 : 0;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
          if (++st == NST) { st = 0; sph ^= 1u; }
        }
        if (!ok) break;
        // rows past the last piece of a short tile
        for (int row = npieces * FT::kPiece + lane; row < kTile; row += 32) {
          convert_row<F>(stage, false, kv, row, cw, scales);
          if (cw == 3) valid_row[row] = 0;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(tile_full);
        if (cw == 0 && lane == 0) TL(1, 5);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;             // TMEM lane quadrant of this warp
    const int myrow = quad * 32 + lane;    // key row (softmax) / output column d (epilogue)
    const int st_tid = tid - 64;           // 0..127
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int bh = butterfly16_head(lane);
    uint32_t ph_t = 0, ph_s = 0, ph_o = 0;
    int redbuf = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
      const ItemInfo it = decode_item<kSparse>(p, item);
      const int ntiles = static_cast<int>((it.n + kTile - 1) / kTile);
      const int h0 = it.hg * kRows;
      const int nh = min(kRows, p.H - h0);
      float m_run[kRows], l_t[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) { m_run[r] = -CUDART_INF_F; l_t[r] = 0.f; }

      for (int t = 0; t < ntiles; ++t) {
        if (st_tid == 0) TL(3, 1);
        bool w = mbar_wait(tile_full, ph_t, abort_flag);
        ph_t ^= 1u;
        w = w && mbar_wait(s_full, ph_s, abort_flag);
        ph_s ^= 1u;
        if (st_tid == 0) TL(3, 2);
        tc_fence_after();
        float s[kRows];
        float4 sc = make_float4(1.f, 1.f, 1.f, 1.f);
        if (F == kDS) {
          float d0[16], d1[16], d2[16], d3[16], dr[16];
          tmem_ld16(tl + 0, d0);
          tmem_ld16(tl + 16, d1);
          tmem_ld16(tl + 32, d2);
          tmem_ld16(tl + 48, d3);
          tmem_ld16(tl + 64, dr);
          tmem_ld_wait();
          sc = *reinterpret_cast<const float4*>(scales + myrow * 4);
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            s[r] = (sc.x * d0[r] + sc.y * d1[r] + sc.z * d2[r] + sc.w * d3[r] + dr[r]) * p.sig2;
        } else {
          float d0[16];
          tmem_ld16(tl, d0);
          tmem_ld_wait();
#pragma unroll
          for (int r = 0; r < kRows; ++r) s[r] = d0[r] * p.sig2;
        }
        if (!valid_row[myrow]) {
#pragma unroll
          for (int r = 0; r < kRows; ++r) s[r] = -CUDART_INF_F;
        }
        // ---- tile max per head across the 128 keys
        float* rb = red + redbuf * 64;
        redbuf ^= 1;
        {
          const float wm = butterfly16<true>(s, lane);
          if ((lane & 1) == 0) rb[quad * 16 + bh] = wm;
        }
        ok = named_bar_and(1, 128, w);
        if (!ok) break;
        bool changed = false;
        float alpha[kRows], pr[kRows];
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const float4 q0 = reinterpret_cast<const float4*>(rb)[r4];
          const float4 q1 = reinterpret_cast<const float4*>(rb + 16)[r4];
          const float4 q2 = reinterpret_cast<const float4*>(rb + 32)[r4];
          const float4 q3 = reinterpret_cast<const float4*>(rb + 48)[r4];
          const float tm[4] = {fmaxf(fmaxf(q0.x, q1.x), fmaxf(q2.x, q3.x)), fmaxf(fmaxf(q0.y, q1.y), fmaxf(q2.y, q3.y)),
                               fmaxf(fmaxf(q0.z, q1.z), fmaxf(q2.z, q3.z)), fmaxf(fmaxf(q0.w, q1.w), fmaxf(q2.w, q3.w))};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 4 * r4 + e;
            const float mnew = fmaxf(m_run[r], tm[e]);
            const float mu = (mnew == -CUDART_INF_F) ? 0.f : mnew;
            alpha[r] = exp2f(m_run[r] - mu);
            pr[r] = exp2f(s[r] - mu);
            l_t[r] = l_t[r] * alpha[r] + pr[r];
            changed |= (mnew != m_run[r]);
            m_run[r] = mnew;
          }
        }
        // ---- PV of the previous tile must be complete before O^T is rescaled and P reused
        if (st_tid == 0) TL(3, 3);
        if (t > 0) {
          w = mbar_wait(o_done, ph_o, abort_flag);
          ph_o ^= 1u;
          tc_fence_after();
          if (st_tid == 0) TL(3, 4);
          if (w && changed) {
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
              float o[16];
              tmem_ld16(tl + kOCol + 16 * j, o);
              tmem_ld_wait();
#pragma unroll
              for (int r = 0; r < kRows; ++r) o[r] *= alpha[r];
              tmem_st16(tl + kOCol + 16 * j, o);
            }
            tmem_st_wait();
          }
        }
        // ---- P^T (MN-major, no swizzle): key row myrow, heads 0..7 | 8..15
        {
          const uint32_t off = (myrow >> 3) * 256 + (myrow & 7) * 16;
          const float f4[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
          for (int j = 0; j < FT::kNP; ++j) {
            const float f = (F == kDS) ? f4[j] : 1.f;
            uint4 lo, hi;
            lo.x = pack2(pr[0] * f, pr[1] * f, F == kBF16);
            lo.y = pack2(pr[2] * f, pr[3] * f, F == kBF16);
            lo.z = pack2(pr[4] * f, pr[5] * f, F == kBF16);
            lo.w = pack2(pr[6] * f, pr[7] * f, F == kBF16);
            hi.x = pack2(pr[8] * f, pr[9] * f, F == kBF16);
            hi.y = pack2(pr[10] * f, pr[11] * f, F == kBF16);
            hi.z = pack2(pr[12] * f, pr[13] * f, F == kBF16);
            hi.w = pack2(pr[14] * f, pr[15] * f, F == kBF16);
            *reinterpret_cast<uint4*>(ps + j * 4096 + off) = lo;
            *reinterpret_cast<uint4*>(ps + j * 4096 + off + 128) = hi;
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = named_bar_and(1, 128, w);
        if (!ok) break;
        if (st_tid == 0) mbar_arrive(p_full);
        if (st_tid == 0) TL(3, 5);
      }
      if (!ok) break;
      bool w = true;
      if (ntiles > 0) {
        w = mbar_wait(o_done, ph_o, abort_flag);
        ph_o ^= 1u;
        tc_fence_after();
      }

      // ---- epilogue: l = sum over the 128 key lanes; O^T lane myrow = output column d
      float* rl = red + 128;
      {
        const float ws = butterfly16<false>(l_t, lane);
        if ((lane & 1) == 0) rl[quad * 16 + bh] = ws;
      }
      ok = named_bar_and(1, 128, w);
      if (!ok) break;
      float inv[kRows], lse_r[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const float l = (rl[r] + rl[16 + r]) + (rl[32 + r] + rl[48 + r]);
        const bool live = (ntiles > 0) && (l > 0.f);
        inv[r] = live ? p.out_scale / l : 0.f;
        lse_r[r] = live ? (m_run[r] + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      }
      const bool final_out = (p.n_splits == 1);
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        float o[16];
        if (ntiles > 0) {
          tmem_ld16(tl + kOCol + 16 * j, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int r = 0; r < kRows; ++r) o[r] = 0.f;
        }
        const int d = 128 * j + myrow;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          if (r < nh) {
            const float val = o[r] * inv[r];
            if (final_out) {
              *reinterpret_cast<__nv_bfloat16*>(p.out + it.row * p.o_s0b + (h0 + r) * p.o_s1b + 2 * d) =
                  __float2bfloat16_rn(val);
            } else {
              p.part_o[((static_cast<int64_t>(it.split) * p.n_rows + it.row) * p.H + h0 + r) * kLora + d] = val;
            }
          }
        }
      }
      if (myrow < nh) {
        float lv = lse_r[0];
#pragma unroll
        for (int r = 1; r < kRows; ++r)
          if (myrow == r) lv = lse_r[r];
        if (final_out) {
          if (p.lse) p.lse[static_cast<int64_t>(it.row) * p.H + h0 + myrow] = lv;
        } else {
          p.part_lse[(static_cast<int64_t>(it.split) * p.n_rows + it.row) * p.H + h0 + myrow] = lv;
        }
      }
      tc_fence_before();
      named_bar_sync(1, 128);   // O^T reads and the reduction buffers are done before the next item
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag == 2) set_device_error(p.err, 16u);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace mla
