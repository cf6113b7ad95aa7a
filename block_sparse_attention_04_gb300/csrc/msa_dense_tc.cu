// Dense causal GQA attention on tensor cores (msa_dense_attn for prefill
// shapes): the full-attention equation of "MiniMax 模型迭代与竞品分析"
// section 2, s = q.k / sqrt(d), softmax over every key j <= t, o = sum a v,
// on the KV-block-major cache of "前沿架构解码手记（三）" section 2.1.  M3
// keeps its first layers dense (section 3 of the first page).
//
// Query-outer: a work item is one 128-query tile of one sequence and a pair
// of query heads of one KV group, run as two chains (one head each) over every
// causal key block, so that both chains' S = Q K^T and O += P V read the same
// K and V block from shared memory.  O stays in tensor memory across the
// blocks (an online softmax); nothing leaves the SM until the item's output.
//   warp 0       TMA of the item's two Q tiles (128 queries x D, one head each)
//   warp 1       TMA of K and V blocks of the group's KV head, 2-deep rings
//   warp 2       tcgen05.mma, per block: P.V(c0, kb-1), S(c0, kb),
//                P.V(c1, kb-1), S(c1, kb); S and P share TMEM columns
//                [128c, 128c + 128), O is at [256 + 128c, ...)
//   warps 3-10   one warpgroup per chain, a query row per thread: row
//                maximum, P = 2^(s - m) as bf16 written over S, row sum; O
//                rescaled in TMEM only when a row's maximum grows by more
//                than 2^8 (until then P may reach 256, exact in bf16 and
//                fp32); at the item's end O / l as bf16 to the output.
#include "msa_device.cuh"
#include "msa_tc.h"
#include "msa_tma.h"

namespace msa {
namespace {

constexpr int kDQWarp = 0, kDKVWarp = 1, kDMmaWarp = 2, kDSoftWarp0 = 3;
constexpr int kDenseThreads = 32 * 11;
constexpr int kDKVStages = 2;
constexpr float kLazyRescale = 8.f;  // log2 of the growth of P tolerated before O is rescaled
constexpr int kDItemRing = 4;        // item ids published by the Q warp, ahead of use
constexpr int kDItemReaders = 10;    // the K/V lane, the MMA warp, the 8 softmax warps

struct DenseArgs {
  Shape s;
  Positions pos;
  int nqt;      // 128-query tiles per sequence
  int npair;    // head pairs per KV group: ceil(H/G / 2)
  int nitems;   // nqt * B * G * npair
  int* next_item;  // shared counter of taken items (zeroed with the status word)
  uint16_t* out;
  int* status;
  uint32_t wait_polls;  // poll cap of the pipeline waits (0: wall-clock bound only)
};

template <int D>
struct DenseCfg {
  static constexpr int kNHalf = D / 64;
  static constexpr int kHalf = 128 * 128;       // one box: 128 rows x 64 dims (16 KiB)
  static constexpr int kTile = kNHalf * kHalf;  // 128 rows x D: a Q tile, a K or a V block
  static constexpr int kSmem = 2 * kTile + 2 * kDKVStages * kTile + 512 + 1024;
  static constexpr uint32_t kTmemCols = 512;
};

// Item it, heaviest first: query tiles from the last (most key blocks) down.
// CTAs take items from a shared counter as they go (greedy list scheduling).
struct DenseItem {
  int b, g, ha, hb, qt, nblk;
  bool hb_real;  // false: the group has an odd head count and chain 1 repeats ha
};

__device__ __forceinline__ DenseItem dense_item(const DenseArgs& a, int it) {
  DenseItem d;
  const int per = a.s.B * a.s.G * a.npair;
  d.qt = a.nqt - 1 - it / per;
  int r = it % per;
  const int pair = r % a.npair;
  r /= a.npair;
  d.g = r % a.s.G;
  d.b = r / a.s.G;
  const int hpg = a.s.H / a.s.G;
  d.ha = d.g * hpg + 2 * pair;
  d.hb_real = 2 * pair + 1 < hpg;
  d.hb = d.hb_real ? d.ha + 1 : d.ha;
  const int i_last = min(a.s.T - 1, d.qt * 128 + 127);
  d.nblk = (int)(((int64_t)a.pos.q_start[d.b] + i_last) / kBlock) + 1;
  return d;
}

template <int D>
__global__ void __launch_bounds__(kDenseThreads, 1)
    dense_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ DenseArgs a) {
  using C = DenseCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;                           // [chain] Q tiles
  uint8_t* sK = sQ + 2 * C::kTile;              // [kDKVStages] K blocks
  uint8_t* sV = sK + kDKVStages * C::kTile;     // [kDKVStages] V blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kDKVStages * C::kTile);
  uint64_t* q_full = bars;                      // both Q tiles of the item landed
  uint64_t* q_empty = q_full + 1;               // the item's last S MMAs are done
  uint64_t* k_full = q_empty + 1;               // kDKVStages
  uint64_t* k_empty = k_full + kDKVStages;
  uint64_t* v_full = k_empty + kDKVStages;
  uint64_t* v_empty = v_full + kDKVStages;
  uint64_t* s_full = v_empty + kDKVStages;      // per chain: S of the block is in TMEM
  uint64_t* p_full = s_full + 2;                // per chain: P written over S (O rescaled)
  uint64_t* o_full = p_full + 2;                // per chain: the item's last P.V is done
  uint64_t* bar_fin = o_full + 2;
  uint64_t* it_full = bar_fin + 1;              // kDItemRing: an item id is published
  uint64_t* it_empty = it_full + kDItemRing;    // kDItemRing: every reader has it
  int* item_ring = reinterpret_cast<int*>(it_empty + kDItemRing);  // ids, -1: no more
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(item_ring + kDItemRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < kDKVStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(&s_full[c], 1);
      mbar_init(&p_full[c], 128);
      mbar_init(&o_full[c], 1);
    }
    mbar_init(bar_fin, 1);
    for (int i = 0; i < kDItemRing; ++i) {
      mbar_init(&it_full[i], 1);
      mbar_init(&it_empty[i], kDItemReaders);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kDMmaWarp) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int T = a.s.T;

  if (warp == kDQWarp) {
    // ------------------------------------------------------- Q TMA (warp 0)
    if (lane == 0) {
      // Takes the items: publishes item k + 1's id (-1 once none is left, or
      // after an abort) before it loads item k's Q, so that the K/V copies
      // of the next item can start during this one.
      const uint64_t pol = l2_policy_evict_first();
      int cur = atomicAdd(a.next_item, 1);
      if (cur >= a.nitems) cur = -1;
      item_ring[0] = cur;
      mbar_arrive(&it_full[0]);
      int k = 0;
      for (; cur >= 0; ++k) {
        const int r = k + 1, slot = r % kDItemRing;
        if (r >= kDItemRing &&
            !mbar_wait(&it_empty[slot], ((r / kDItemRing) - 1) & 1, a.status, a.wait_polls)) {
          *abort_flag = 1;
          break;
        }
        int nx = *abort_flag ? a.nitems : atomicAdd(a.next_item, 1);
        if (nx >= a.nitems) nx = -1;
        item_ring[slot] = nx;
        mbar_arrive(&it_full[slot]);
        const DenseItem d = dense_item(a, cur);
        if (k > 0 && !mbar_wait(q_empty, (k - 1) & 1, a.status, a.wait_polls)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * C::kTile);
        const int z = d.b * T + d.qt * 128;
#pragma unroll
        for (int h = 0; h < C::kNHalf; ++h) {
          tma_load_3d_hint(smem_u32(sQ + h * C::kHalf), &tm_q, q_full, h * 64, d.ha, z, pol);
          tma_load_3d_hint(smem_u32(sQ + C::kTile + h * C::kHalf), &tm_q, q_full, h * 64, d.hb, z,
                           pol);
        }
        cur = nx;
      }
      // no copy may still be landing when the CTA exits
      if (k > 0) mbar_wait(q_full, (k - 1) & 1, nullptr);
    }
  } else if (warp == kDKVWarp) {
    // ----------------------------------------------------- K/V TMA (warp 1)
    if (lane == 0) {
      int n = 0;
      bool ok = true, k_only = false;  // k_only: step n's K is loaded, its V is not
      for (int ki = 0; ok && !*abort_flag; ++ki) {
        const int slot = ki % kDItemRing;
        if (!mbar_wait(&it_full[slot], (ki / kDItemRing) & 1, a.status, a.wait_polls)) {
          ok = false;
          break;
        }
        const int it = item_ring[slot];
        mbar_arrive(&it_empty[slot]);
        if (it < 0) break;
        const DenseItem d = dense_item(a, it);
        for (int kb = 0; kb < d.nblk; ++kb, ++n) {
          const int ks = n % kDKVStages;
          const uint32_t w = (uint32_t)(n / kDKVStages);
          // through the block table when the caches are paged; an entry
          // outside the pool (flagged) reads zeros from past the pool's end
          const int64_t pb = cache_block(a.s, d.b, kb, a.status);
          const int row = (int)((pb < 0 ? a.s.cache_blocks() : pb) * kBlock);
          if (!mbar_wait(&k_empty[ks], (w & 1) ^ 1, a.status, a.wait_polls)) { ok = false; break; }
          mbar_arrive_expect_tx(&k_full[ks], C::kTile);
#pragma unroll
          for (int h = 0; h < C::kNHalf; ++h)
            tma_load_3d(smem_u32(sK + ks * C::kTile + h * C::kHalf), &tm_k, &k_full[ks], h * 64, d.g,
                        row);
          if (!mbar_wait(&v_empty[ks], (w & 1) ^ 1, a.status, a.wait_polls)) {
            ok = false;
            k_only = true;
            break;
          }
          mbar_arrive_expect_tx(&v_full[ks], C::kTile);
#pragma unroll
          for (int h = 0; h < C::kNHalf; ++h)
            tma_load_3d(smem_u32(sV + ks * C::kTile + h * C::kHalf), &tm_v, &v_full[ks], h * 64, d.g,
                        row);
        }
      }
      if (!ok) *abort_flag = 1;
      // no copy may still be landing when the CTA exits: the last load of
      // each ring slot (a V load is issued only after its slot's K load)
      for (int m = n - 1; m >= 0 && m >= n - kDKVStages; --m) {
        const int ks = m % kDKVStages;
        const uint32_t ph = (uint32_t)(m / kDKVStages) & 1;
        mbar_wait(&k_full[ks], ph, nullptr);
        mbar_wait(&v_full[ks], ph, nullptr);
      }
      if (k_only) mbar_wait(&k_full[n % kDKVStages], (uint32_t)(n / kDKVStages) & 1, nullptr);
    }
  } else if (warp == kDMmaWarp) {
    // ---------------------------------------------------------- MMA (warp 2)
    // The whole warp runs the loop; one elected lane issues and commits.
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
    const uint64_t qdesc0 = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
    const uint64_t kdesc0 = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
    const uint64_t vdesc0 = smem_desc(smem_u32(sV), C::kHalf, 1024, kSwizzle128B);
    int n = 0, k = 0;
    bool ok = true;
    for (; ok; ++k) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      const int slot = k % kDItemRing;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&it_full[slot], (k / kDItemRing) & 1, a.status, a.wait_polls));
      if (!ok) break;
      // every lane's read of the slot is consumed (by the shuffle) before the
      // slot is handed back, so no read can still be pending when it is rewritten
      const int it = __shfl_sync(0xffffffffu, item_ring[slot], 0);
      if (lane == 0) mbar_arrive(&it_empty[slot]);
      if (it < 0) break;
      const DenseItem d = dense_item(a, it);
      ok = __all_sync(0xffffffffu, mbar_wait(q_full, k & 1, a.status, a.wait_polls));
      if (!ok) break;
      int pks = 0;
      uint32_t pw = 0;
      for (int kb = 0; kb <= d.nblk && ok; ++kb) {
        const bool has_s = kb < d.nblk;
        const int ks = n % kDKVStages;
        const uint32_t w = (uint32_t)(n / kDKVStages);
        bool okl = !has_s || mbar_wait(&k_full[ks], w & 1, a.status, a.wait_polls);
        if (kb > 0) okl = okl && mbar_wait(&v_full[pks], pw & 1, a.status, a.wait_polls);
        ok = __all_sync(0xffffffffu, okl);
        if (!ok) break;
        for (int c = 0; c < 2; ++c) {
          if (kb > 0) {
            // ---- P.V(c, kb - 1): P in TMEM columns [128c, 128c + 64)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&p_full[c], (uint32_t)(n - 1) & 1, a.status, a.wait_polls));
            if (!ok) break;
            tc_fence_after();
            const uint64_t vd = vdesc0 + (uint64_t)((pks * C::kTile) >> 4);
            if (elect_one()) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                tc_mma_f16_ts(tmem + 256 + c * 128, tmem + c * 128 + j * 8,
                              vd + (uint64_t)((j * 2048) >> 4), idesc_o, (kb > 1 || j > 0) ? 1u : 0u);
              if (!has_s) tc_commit(&o_full[c]);
              if (c == 1) tc_commit(&v_empty[pks]);
            }
            __syncwarp();
          }
          if (has_s) {
            // ---- S(c, kb) = Q_c K_kb^T
            tc_fence_after();
            const uint64_t qd = qdesc0 + (uint64_t)((c * C::kTile) >> 4);
            const uint64_t kd = kdesc0 + (uint64_t)((ks * C::kTile) >> 4);
            if (elect_one()) {
#pragma unroll
              for (int j = 0; j < D / 16; ++j)  // 16 dims: (j & 3) * 32 bytes within a 64-dim half
                tc_mma_f16(tmem + c * 128,
                           qd + (uint64_t)(((j >> 2) * C::kHalf + (j & 3) * 32) >> 4),
                           kd + (uint64_t)(((j >> 2) * C::kHalf + (j & 3) * 32) >> 4), idesc_s,
                           j > 0 ? 1u : 0u);
              tc_commit(&s_full[c]);
              if (c == 1) {
                tc_commit(&k_empty[ks]);
                if (kb + 1 == d.nblk) tc_commit(q_empty);
              }
            }
            __syncwarp();
          }
        }
        if (has_s) {
          pks = ks;
          pw = w;
          ++n;
        }
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
    // all MMAs done before TMEM is released
    if (elect_one()) tc_commit(bar_fin);
    __syncwarp();
    mbar_wait(bar_fin, 0, nullptr);
  } else {
    // ------------------------------------- softmax + output (warps 3-10)
    const int c = (warp - kDSoftWarp0) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t s_base = tmem + ((uint32_t)(quad * 32) << 16) + c * 128;
    const uint32_t o_base = tmem + ((uint32_t)(quad * 32) << 16) + 256 + c * 128;
    const float sl = a.s.scale * kLog2e;
    int n = 0, k = 0;
    bool ok = true;
    for (; ok; ++k) {
      const int slot = k % kDItemRing;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&it_full[slot], (k / kDItemRing) & 1, a.status, a.wait_polls))) {
        ok = false;
        break;
      }
      // every lane's read of the slot is consumed (by the shuffle) before the
      // slot is handed back, so no read can still be pending when it is rewritten
      const int it = __shfl_sync(0xffffffffu, item_ring[slot], 0);
      if (lane == 0) mbar_arrive(&it_empty[slot]);
      if (it < 0) break;
      const DenseItem d = dense_item(a, it);
      const int i = d.qt * 128 + r;
      const bool valid = i < T && (c == 0 || d.hb_real);
      const int64_t tq = (int64_t)a.pos.q_start[d.b] + i;
      float m_ref = -INFINITY, l = 0.f;
      for (int kb = 0; kb < d.nblk; ++kb, ++n) {
        if (__any_sync(0xffffffffu, *abort_flag != 0) ||
            !__all_sync(0xffffffffu, mbar_wait(&s_full[c], (uint32_t)n & 1, a.status, a.wait_polls))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // tokens kb*128 + col with col > lim are masked (the last blocks only)
        const int64_t lim64 = tq - (int64_t)kb * kBlock;
        const int lim = lim64 > kBlock ? kBlock : (int)lim64;
        const bool masked = __any_sync(0xffffffffu, lim < kBlock - 1);
        // pass 1: row maximum of the scaled scores (with a negative scale,
        // the minimum of the raw ones); away from the diagonal the load
        // reduces its 16 scores itself
        float mx = -INFINITY;
        if (masked) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t h[16];
            tmem_ld16(s_base + cc * 16, h);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float x = __uint_as_float(h[e]) * sl;
              mx = fmaxf(mx, cc * 16 + e <= lim ? x : -INFINITY);
            }
          }
        } else if (sl >= 0.f) {
          float r = -INFINITY;
#pragma unroll 1
          for (int cc = 0; cc < 8; cc += 2) {
            const float r0 = tmem_ld16_red<true>(s_base + cc * 16);
            const float r1 = tmem_ld16_red<true>(s_base + cc * 16 + 16);
            tmem_ld_wait();
            r = fmax3(r, r0, r1);
          }
          mx = r * sl;
        } else {
          float r = INFINITY;
#pragma unroll 1
          for (int cc = 0; cc < 8; cc += 2) {
            const float r0 = tmem_ld16_red<false>(s_base + cc * 16);
            const float r1 = tmem_ld16_red<false>(s_base + cc * 16 + 16);
            tmem_ld_wait();
            r = fmin3(r, r0, r1);
          }
          mx = r * sl;
        }
        // lazy rescale: a new reference maximum only when the row maximum
        // grew by more than kLazyRescale (always on the first block)
        const bool grow = mx > m_ref + kLazyRescale;
        float alpha = 1.f;
        if (grow) {
          alpha = ex2(m_ref - mx);  // 0 on the first block (m_ref = -inf)
          m_ref = mx;
          l *= alpha;
        }
        // O of the earlier blocks times alpha, in TMEM (the P.V of block
        // kb - 1 is done: the S of block kb was issued after it)
        if (kb > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 16; ++cc) {
            uint32_t h[16];
            tmem_ld16(o_base + cc * 16, h);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) h[e] = __float_as_uint(__uint_as_float(h[e]) * alpha);
            tmem_st16(o_base + cc * 16, h);
          }
        }
        // pass 2: P = 2^(x - m_ref) as bf16, two per column, written over S
        // (the 32 scores of columns [32cc, 32cc + 32) are read before columns
        // [16cc, 16cc + 16), already read, are written); row sum
        // The FMA pipe is the busier one here: the scaling and the sums use
        // packed two-lane instructions, and every exponential goes to the MUFU
        // unit (measured at 32K: moving 2, 4 or 6 of 16 pairs to the FMA-pipe
        // polynomial cost 5, 11 and 21 %).
        const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(-m_ref, -m_ref);
        float2 lsum = make_float2(0.f, 0.f);
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t wv[16];
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t h[16];
            tmem_ld16(s_base + cc * 32 + hf * 16, h);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int col = cc * 32 + hf * 16 + 2 * u;
              const float2 x =
                  ffma2(make_float2(__uint_as_float(h[2 * u]), __uint_as_float(h[2 * u + 1])), sl2, nm2);
              float2 pp = make_float2(ex2(x.x), ex2(x.y));
              if (masked) {
                pp.x = col <= lim ? pp.x : 0.f;
                pp.y = col + 1 <= lim ? pp.y : 0.f;
              }
              lsum = fadd2(lsum, pp);
              wv[hf * 8 + u] = pack_bf16(pp.x, pp.y);
            }
          }
          tmem_st16(s_base + cc * 16, wv);
        }
        l += lsum.x + lsum.y;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[c]);
      }
      if (!ok) break;
      // output: O / l after the item's last P.V
      if (!__all_sync(0xffffffffu, mbar_wait(&o_full[c], (uint32_t)k & 1, a.status, a.wait_polls))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = 1.f / l;
      uint16_t* dst =
          a.out + (((size_t)d.b * T + (valid ? i : 0)) * a.s.H + (c == 0 ? d.ha : d.hb)) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 16; ++cc) {
        uint32_t h[16];
        tmem_ld16(o_base + cc * 16, h);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int e8 = 0; e8 < 2; ++e8) {
            uint4 pk;
            pk.x = pack_bf16(__uint_as_float(h[e8 * 8 + 0]) * inv, __uint_as_float(h[e8 * 8 + 1]) * inv);
            pk.y = pack_bf16(__uint_as_float(h[e8 * 8 + 2]) * inv, __uint_as_float(h[e8 * 8 + 3]) * inv);
            pk.z = pack_bf16(__uint_as_float(h[e8 * 8 + 4]) * inv, __uint_as_float(h[e8 * 8 + 5]) * inv);
            pk.w = pack_bf16(__uint_as_float(h[e8 * 8 + 6]) * inv, __uint_as_float(h[e8 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + cc * 16 + e8 * 8) = pk;
          }
        }
      }
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kDMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_dense_tc_impl(const Shape& s, const Positions& pos, const uint16_t* q,
                                 const uint16_t* k, const uint16_t* v, uint16_t* out, int* status,
                                 cudaStream_t st) {
  using C = DenseCfg<D>;
  // the item counter sits in the word after the status word; both are zeroed
  if (cudaMemsetAsync(status, 0, 2 * sizeof(int), st) != cudaSuccess) return cudaErrorUnknown;
  CUtensorMap tm_q, tm_k, tm_v;
  {
    // q as (D dims, H heads, B*T queries): one box = 128 queries x 64 dims
    // of one head
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)s.H, (cuuint64_t)s.B * s.T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)s.H * D * 2};
    cuuint32_t box[3] = {64, 1, 128};
    if (!encode_bf16_map(&tm_q, q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)s.G, (cuuint64_t)(s.cache_blocks() * kBlock)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)s.G * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kBlock};
    if (!encode_bf16_map(&tm_k, k, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_map(&tm_v, v, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  DenseArgs a;
  a.s = s;
  a.pos = pos;
  a.nqt = (s.T + 127) / 128;
  a.npair = (s.H / s.G + 1) / 2;
  a.nitems = a.nqt * s.B * s.G * a.npair;
  a.next_item = status + 1;
  a.out = out;
  a.status = status;
  a.wait_polls = debug_wait_polls();
  cudaError_t e = cudaFuncSetAttribute(dense_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int ctas = sm_count();
  const int grid = a.nitems < ctas ? a.nitems : ctas;
  note_launches(1);
  dense_tc_kernel<D><<<grid, kDenseThreads, C::kSmem, st>>>(tm_q, tm_k, tm_v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_tc(const Shape& s, const Positions& pos, const uint16_t* q,
                            const uint16_t* k, const uint16_t* v, uint16_t* out, int* status,
                            cudaStream_t st) {
  if (s.B == 0 || s.T == 0) return cudaSuccess;
  return s.D == 128 ? launch_dense_tc_impl<128>(s, pos, q, k, v, out, status, st)
                    : launch_dense_tc_impl<64>(s, pos, q, k, v, out, status, st);
}

}  // namespace msa
