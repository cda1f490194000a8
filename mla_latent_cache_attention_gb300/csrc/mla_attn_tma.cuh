// mla_attn_tma.cuh -- paged MLA decode over the bf16 cache with TMA page loads.
//
// Same computation as mla_attn_kernel (swap-AB tcgen05 MMAs: QK with M = 128 keys, N = 16
// heads; PV with M = 128 latent columns), but the key tile is loaded by the tensor memory
// accelerator straight from the paged cache: a 3-D tensor map [num_blocks][block_size][1152 B]
// with 128-byte swizzle and boxes of 128 bytes x BR rows, so every box lands in the
// canonical operand layout of one 64-wide block and no thread touches the data on its way
// to the tensor core.  (A gather probe on GB300 moved 656-byte records at 2.3 TB/s with one
// bulk copy per record and at 6.7 TB/s with page boxes.)
//
// The 128-key tile is split into five load groups -- block pairs {0,1}, {2,3}, {4,5}, {6,7}
// and block 8 -- each with its own barrier.  QK of a tile starts as soon as its first pair has
// landed; the next tile's block 8 is reloaded once QK is done with it, and pair j once PV
// tile j is done with it, so loads overlap the MMAs.  The tile after the current one is
// prefetched into L2 as soon as its page ids are known.
//
// Warps: 0 producer (lane 0 issues the TMA, the lanes resolve page ids), 1 MMA issuer and TMEM
// owner, 2..5 softmax + epilogue (they also zero the rows of keys past the end of a tile, so
// that stale rows can never reach PV).
#pragma once
#include <cuda.h>

#include "mla_attn.cuh"

namespace mla {

constexpr int kTmaThreads = 192;

struct TmaSmem {
  static constexpr int kKV = 0;
  static constexpr int kQ = kKV + kBlk * kBlkBytes;
  static constexpr int kP = kQ + kBlk * kQBlkBytes;
  static constexpr int kRed = kP + 4096;                // [2][4][16] + [4][16] fp32
  static constexpr int kMeta = kRed + 3 * 4 * 16 * 4;   // per tile parity: valid-page mask, keys in tile
  static constexpr int kBar = kMeta + 64;
  static constexpr int kNumBars = 5 + 4 + 4;            // kv_full[5], pair_free[4], s_full, p_full, q_full, final
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= kSmemLimit, "shared memory budget");
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* tm, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tm), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}

// Work cursor over this CTA's (item, tile) pairs, skipping items without keys.
struct TileCursor {
  int item, t, ntiles;
  ItemInfo it;
};

__device__ __forceinline__ TileCursor cursor_from(const AttnParams& p, int item) {
  TileCursor c{item, 0, 0, ItemInfo{}};
  for (; c.item < p.n_items; c.item += gridDim.x) {
    c.it = decode_item<false>(p, c.item);
    c.ntiles = static_cast<int>((c.it.n + kTile - 1) / kTile);
    if (c.ntiles > 0) return c;
  }
  return c;
}
__device__ __forceinline__ TileCursor cursor_next(const AttnParams& p, const TileCursor& c) {
  if (c.t + 1 < c.ntiles) {
    TileCursor n = c;
    n.t += 1;
    return n;
  }
  return cursor_from(p, c.item + gridDim.x);
}

// Page q of the cursor's tile: rows q*BR .. q*BR+BR-1 of the tile.  Returns the block id
// (or -1 when the page holds no key of the item or its id is out of range) and the row offset
// of the page's first key inside its block.
__device__ __forceinline__ int64_t tile_page(const AttnParams& p, const TileCursor& c, int q, int& y,
                                             uint32_t& errbits) {
  const int BR = p.tma_rows;
  const int64_t pos = c.it.k0 + static_cast<int64_t>(c.t) * kTile + static_cast<int64_t>(q) * BR;
  y = 0;
  if (pos >= c.it.k0 + c.it.n) return -1;
  const int b = c.it.row / p.q_len;
  const int64_t blk = p.block_table[static_cast<int64_t>(b) * p.bt_stride + pos / p.block_size];
  if (blk < 0 || blk >= p.num_blocks) {
    errbits |= 2u;
    return -1;
  }
  y = static_cast<int>(pos % p.block_size);
  return blk;
}

__global__ void __launch_bounds__(kTmaThreads, 1)
    mla_attn_tma_bf16_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm) {
  using SM = TmaSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem + SM::kKV;
  uint8_t* qs = smem + SM::kQ;
  uint8_t* ps = smem + SM::kP;
  float* red = reinterpret_cast<float*>(smem + SM::kRed);
  uint32_t* tmeta = reinterpret_cast<uint32_t*>(smem + SM::kMeta);   // [2] {page mask, keys}
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBar);
  uint64_t* kv_full = bars;          // [5]: pairs 0..3, block 8
  uint64_t* pair_free = bars + 5;    // [4]: PV tile j done (pair_free[3] = all MMAs of the tile done)
  uint64_t* s_full = bars + 9;
  uint64_t* p_full = bars + 10;
  uint64_t* q_full = bars + 11;
  uint64_t* mma_final = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BR = p.tma_rows;
  const int NPG = kTile / BR;      // pages per tile (BR divides 128)
  TL_DECL;

  if (tid == 0) {
    for (int g = 0; g < 5; ++g) mbar_init(&kv_full[g], 1);
    for (int j = 0; j < 4; ++j) mbar_init(&pair_free[j], 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 1);
    mbar_init(q_full, 1);
    mbar_init(mma_final, 1);
    *abort_flag = 0;
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

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    uint32_t errbits = 0;
    uint32_t ph_s = 0, ph_pf = 0;
    bool ok = true;
    int g = 0;     // tile counter of this CTA
    bool armed = false;
    uint32_t armed_par = 0;
    TileCursor cur = cursor_from(p, blockIdx.x);
    // page ids of the current tile (lane q < NPG holds page q)
    int y_c = 0;
    int64_t blk_c = (cur.item < p.n_items && lane < NPG) ? tile_page(p, cur, lane, y_c, errbits) : -1;
    while (ok && cur.item < p.n_items) {
      const TileCursor nxt = cursor_next(p, cur);
      int y_n = 0;
      const int64_t blk_n = (nxt.item < p.n_items && lane < NPG) ? tile_page(p, nxt, lane, y_n, errbits) : -1;
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, lane < NPG && blk_c >= 0);
      const int npages = __popc(mask);
      if (lane == 0) {
        tmeta[2 * (g & 1)] = mask;
        tmeta[2 * (g & 1) + 1] = static_cast<uint32_t>(tile_keys(cur.it.n, cur.t));
      }
      // groups in the order their buffers free up: block 8 (after QK), then pairs 0..3 (after PV j)
      if (lane == 0) TL(0, 1);
      for (int gi = 0; gi < 5 && ok; ++gi) {
        const int grp = (gi == 0) ? 4 : gi - 1;
        if (g > 0) {
          bool w;
          if (grp == 4) {
            w = mbar_wait(s_full, ph_s, abort_flag);
            ph_s ^= 1u;
          } else {
            w = mbar_wait(&pair_free[grp], ph_pf, abort_flag);
            if (grp == 3) ph_pf ^= 1u;
          }
          if (!w) { ok = false; break; }
        }
        const int nblk = (grp == 4) ? 1 : 2;
        if (lane == 0) mbar_arrive_expect_tx(&kv_full[grp], static_cast<uint32_t>(npages * nblk * BR * 128));
        __syncwarp();
        for (int q = 0; q < NPG; ++q) {
          const int64_t blk = __shfl_sync(0xFFFFFFFFu, blk_c, q);
          const int y = __shfl_sync(0xFFFFFFFFu, y_c, q);
          if (lane == 0 && blk >= 0) {
            for (int bb = 0; bb < nblk; ++bb) {
              const int b = (grp == 4) ? 8 : 2 * grp + bb;
              tma_load_3d(kv + b * kBlkBytes + q * BR * 128, &tm, 128 * b, y, static_cast<int>(blk), &kv_full[grp]);
            }
          }
        }
        armed = true;
        armed_par = static_cast<uint32_t>(g & 1);
        if (lane == 0) TL(0, 10 + grp);
      }
      if (!ok) break;
      // L2 prefetch of the next tile
      for (int q = 0; q < NPG; ++q) {
        const int64_t blk = __shfl_sync(0xFFFFFFFFu, blk_n, q);
        const int y = __shfl_sync(0xFFFFFFFFu, y_n, q);
        if (lane < kBlk && blk >= 0) tma_prefetch_3d(&tm, 128 * lane, y, static_cast<int>(blk));
      }
      blk_c = blk_n;
      y_c = y_n;
      cur = nxt;
      ++g;
    }
    if (armed) {    // never leave TMA loads in flight behind us
      volatile int no_abort = 0;
      for (int grp = 0; grp < 5; ++grp) mbar_wait(&kv_full[grp], armed_par, &no_abort);
    }
    errbits = __reduce_or_sync(0xFFFFFFFFu, errbits);
    if (lane == 0 && errbits) set_device_error(p.err, errbits);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t kv_a = smem_u32(kv), q_a = smem_u32(qs), p_a = smem_u32(ps);
      const uint64_t dK = smem_desc(kv_a, 16, 1024, kSwizzle128B);
      const uint64_t dQ = smem_desc(q_a, 16, 1024, kSwizzle128B);
      const uint64_t dV = smem_desc(kv_a, kBlkBytes, 1024, kSwizzle128B);
      const uint64_t dP = smem_desc(p_a, 256, 128, kSwizzleNone);
      constexpr uint32_t kIdQk = idesc_f16(128, kRows, 1, 1, 0, 0);
      constexpr uint32_t kIdPv = idesc_f16(128, kRows, 1, 1, 1, 1);
      uint32_t ph_kv = 0, ph_p = 0, ph_q = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const ItemInfo it = decode_item<false>(p, item);
        const int ntiles = static_cast<int>((it.n + kTile - 1) / kTile);
        if (ntiles == 0) continue;
        if (!mbar_wait(q_full, ph_q, abort_flag)) { ok = false; break; }
        ph_q ^= 1u;
        for (int t = 0; t < ntiles && ok; ++t) {
          TL(2, 1);
#pragma unroll
          for (int grp = 0; grp < 5; ++grp) {
            if (!mbar_wait(&kv_full[grp], ph_kv, abort_flag)) { ok = false; break; }
            TL(2, 10 + grp);
            tc_fence_after();
            const int b0 = (grp == 4) ? 8 : 2 * grp;
            const int nks = (grp == 4) ? 4 : 8;
#pragma unroll
            for (int kk = 0; kk < nks; ++kk) {
              const int b = b0 + (kk >> 2);
              const uint32_t ko = (kk & 3) * 32;
              mma_f16_ss(tmem, dK + ((b * kBlkBytes + ko) >> 4), dQ + ((b * kQBlkBytes + ko) >> 4), kIdQk,
                         (grp > 0 || kk > 0) ? 1u : 0u);
            }
          }
          if (!ok) break;
          ph_kv ^= 1u;
          mma_commit(s_full);
          TL(2, 2);
          if (!mbar_wait(p_full, ph_p, abort_flag)) { ok = false; break; }
          TL(2, 3);
          ph_p ^= 1u;
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t a = dV + ((2 * j * kBlkBytes + kk * 2048) >> 4);
              const uint64_t b = dP + ((kk * 512) >> 4);
              mma_f16_ss(tmem + kOCol + 16 * j, a, b, kIdPv, (t > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&pair_free[j]);
          }
          TL(2, 4);
        }
      }
      mma_commit(mma_final);
      volatile int no_abort = 0;
      mbar_wait(mma_final, 0, &no_abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;
    const int myrow = quad * 32 + lane;
    const int st_tid = tid - 64;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int bh = butterfly16_head(lane);
    uint32_t ph_s = 0, ph_o = 0, ph_k = 0;
    int redbuf = 0, g = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
      const ItemInfo it = decode_item<false>(p, item);
      const int ntiles = static_cast<int>((it.n + kTile - 1) / kTile);
      const int h0 = it.hg * kRows;
      const int nh = min(kRows, p.H - h0);
      if (ntiles > 0) {
        // query tile (the previous item's last QK is complete: its PV was waited for)
        for (int i = st_tid; i < kRows * 72; i += 128) {
          const int r = i / 72, rem = i % 72, b = rem >> 3, c = rem & 7;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < nh) v = query_chunk<kBF16>(p.q + it.row * p.q_s0b + (h0 + r) * p.q_s1b, b, c);
          *reinterpret_cast<uint4*>(qs + b * kQBlkBytes + sw128(r, c)) = v;
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (st_tid == 0) mbar_arrive(q_full);
      }
      float m_run[kRows], l_t[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) { m_run[r] = -CUDART_INF_F; l_t[r] = 0.f; }

      for (int t = 0; t < ntiles; ++t, ++g) {
        bool w = mbar_wait(&kv_full[4], ph_k, abort_flag);     // tile meta is published with block 8
        ph_k ^= 1u;
        w = w && mbar_wait(s_full, ph_s, abort_flag);
        ph_s ^= 1u;
        tc_fence_after();
        if (st_tid == 0) TL(3, 1);
        const uint32_t pmask = tmeta[2 * (g & 1)];
        const int nk = static_cast<int>(tmeta[2 * (g & 1) + 1]);
        const bool valid = (myrow < nk) && ((pmask >> (myrow / BR)) & 1u);
        float s[kRows];
        {
          float d0[16];
          tmem_ld16(tl, d0);
          tmem_ld_wait();
#pragma unroll
          for (int r = 0; r < kRows; ++r) s[r] = valid ? d0[r] * p.sig2 : -CUDART_INF_F;
        }
        // rows that hold no key of this item never reach PV with stale contents
        if (!valid) {
#pragma unroll
          for (int b = 0; b < 8; ++b)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(kv + b * kBlkBytes + myrow * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
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
          const float tm4[4] = {fmaxf(fmaxf(q0.x, q1.x), fmaxf(q2.x, q3.x)), fmaxf(fmaxf(q0.y, q1.y), fmaxf(q2.y, q3.y)),
                                fmaxf(fmaxf(q0.z, q1.z), fmaxf(q2.z, q3.z)), fmaxf(fmaxf(q0.w, q1.w), fmaxf(q2.w, q3.w))};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 4 * r4 + e;
            const float mnew = fmaxf(m_run[r], tm4[e]);
            const float mu = (mnew == -CUDART_INF_F) ? 0.f : mnew;
            alpha[r] = exp2f(m_run[r] - mu);
            pr[r] = exp2f(s[r] - mu);
            l_t[r] = l_t[r] * alpha[r] + pr[r];
            changed |= (mnew != m_run[r]);
            m_run[r] = mnew;
          }
        }
        if (st_tid == 0) TL(3, 2);
        if (t > 0) {
          w = mbar_wait(&pair_free[3], ph_o, abort_flag);    // PV of the previous tile complete
          ph_o ^= 1u;
          tc_fence_after();
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
        {
          const uint32_t off = (myrow >> 3) * 256 + (myrow & 7) * 16;
          uint4 lo, hi;
          lo.x = pack2(pr[0], pr[1], true);
          lo.y = pack2(pr[2], pr[3], true);
          lo.z = pack2(pr[4], pr[5], true);
          lo.w = pack2(pr[6], pr[7], true);
          hi.x = pack2(pr[8], pr[9], true);
          hi.y = pack2(pr[10], pr[11], true);
          hi.z = pack2(pr[12], pr[13], true);
          hi.w = pack2(pr[14], pr[15], true);
          *reinterpret_cast<uint4*>(ps + off) = lo;
          *reinterpret_cast<uint4*>(ps + off + 128) = hi;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = named_bar_and(1, 128, w);
        if (!ok) break;
        if (st_tid == 0) mbar_arrive(p_full);
        if (st_tid == 0) TL(3, 3);
      }
      if (!ok) break;
      bool w = true;
      if (st_tid == 0) TL(3, 5);
      if (ntiles > 0) {
        w = mbar_wait(&pair_free[3], ph_o, abort_flag);
        ph_o ^= 1u;
        tc_fence_after();
      }
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
      if (st_tid == 0) TL(3, 6);
      tc_fence_before();
      named_bar_sync(1, 128);
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
