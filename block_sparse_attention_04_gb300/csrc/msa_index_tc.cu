// Tensor-core index scan for prefill: steps 1-3 of "MiniMax 模型迭代与竞品分析"
// section 2 (global index scoring over the causal context, 128-token block
// max-pooling, top-16 with the local block forced in) for many queries at once.
//
// Rows are (query, group) pairs, r = (b*T + i)*G + g, so one Q_idx tile of
// 128 rows is 128/G queries x G groups and every group reuses the same K_idx
// tile.  One work item = one row tile x one split of at most kSplitBlocks
// key blocks; a one-CTA pre-pass lists the items that have key blocks,
// heaviest first, and each CTA takes the next item from a shared counter
// whenever it starts one (greedy list scheduling: over the 128 calls of the
// 1M chunked prefill the busiest CTA carries about 2 % more than the mean
// instead of about 10 % with a fixed round-robin deal).  Per item and pair of key
// blocks (256 keys, one MMA of N 256 per 16 dims: a tcgen05.mma costs a fixed
// issue time, so each one is made large):
//   warp 0      TMA: the Q_idx tile once per item, K_idx block pairs through a
//               kStages-deep shared-memory ring;
//   warp 1      tcgen05.mma (M 128, N 256, K Di, bf16 in, fp32 accumulate)
//               into one of two TMEM accumulator stages;
//   warps 2-17  epilogue, four warpgroups: two read each accumulator stage
//               (one key block each), stages alternate between the two
//               pairs; reducing tcgen05.ld of the row's 128 fp32 scores in
//               16-column chunks (the load returns each chunk's maximum),
//               block maximum, insertion into a
//               register-resident top-15 (score desc, block id asc); at
//               the end of the item the four lists of a row merge in one
//               parallel step (each candidate's rank among the 60).
// The [query x block] score matrix never leaves TMEM/registers.  Each item
// writes its rows' partial top-15 lists; the streaming path's k-way merge
// (topk_merge) adds the local block and sorts.
#include <climits>

#include "msa_device.cuh"
#include "msa_tc.h"
#include "msa_tma.h"

namespace msa {
namespace {

constexpr int kTileRows = 128;
constexpr int kItemRows = kTileRows;   // (query, group) rows per work item
constexpr int kSplitBlocks = 1024;
constexpr int kPairKeys = 2 * kBlock;  // keys per MMA (N) and per accumulator stage
constexpr int kStages = 4;             // K_idx stages (two key blocks each) in flight
constexpr int kAccStages = 2;          // TMEM accumulator stages of kPairKeys columns
constexpr int kEpiWarps = 16;          // 4 warpgroups
constexpr int kEpiLists = kEpiWarps / 4;  // ranked lists per row at an item's end: one per warpgroup
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue
constexpr uint32_t kTmemCols = 512;
constexpr int kItemRing = 4;           // item ids published by the copy thread, ahead of use

template <int DI>
struct IdxCfg {
  static constexpr int kRowBytes = DI * 2;
  static constexpr int kBoxBytes = kBlock * kRowBytes;     // one key block of K_idx
  static constexpr int kTileBytes = kTileRows * kRowBytes;  // one Q_idx row tile
  static constexpr int kStageBytes = 2 * kBoxBytes;         // two key blocks
  static constexpr uint32_t kSwz = DI == 64 ? kSwizzle128B : kSwizzle64B;
  static constexpr uint32_t kSbo = 8 * kRowBytes;  // one 8-row swizzle atom
  static constexpr int kKSteps = DI / 16;
  static constexpr int kSmemA = 2 * kTileBytes;             // 2 buffers
  static constexpr int kSmemB = kStages * kStageBytes;
  static constexpr int kSmemX = kEpiLists * kTileRows * kCand * 8;  // the lists at an item's end
  static constexpr int kSmemBar = 512;
  static constexpr int kSmem = kSmemA + kSmemB + kSmemX + kSmemBar + 1024;  // + alignment
};

struct IndexTcArgs {
  Shape s;
  Positions pos;
  int npairs;         // row tiles per sequence
  int nsplit;         // splits per row tile (the merge's list count per row)
  int64_t cap;        // K_idx rows per sequence
  const int2* items;     // (row tile, b << 7 | split), heaviest first
  const int32_t* nitems;
  int32_t* next_item;    // shared counter of taken items (zeroed by the pre-pass)
  Cand* cand;
  int* status;
  uint32_t wait_polls;   // poll cap of the pipeline waits (0: wall-clock bound only)
};

// A work item: the row tile in a word of its own (it reaches T*G/128, which
// the host bounds only by T*G < 2^31), then the sequence (8 bits, B <= 256)
// and the split (7 bits, at most 32 splits of 1024 blocks).
__host__ __device__ __forceinline__ int2 pack_item(int b, int p, int sp) {
  return make_int2(p, (b << 7) | sp);
}

__device__ __forceinline__ int pair_kb_end(const Shape& s, const Positions& pos, int b, int p) {
  const int i_last = min(s.T - 1, ((p + 1) * kItemRows - 1) / s.G);
  return (int)(((int64_t)pos.q_start[b] + i_last) / kBlock);
}

// Dense list of the work items that have key blocks, heaviest first: row
// tiles in descending order (their key ranges grow), each tile's splits in order.
__global__ void __launch_bounds__(1024) index_items_kernel(Shape s, Positions pos, int npairs,
                                                           int2* items, int32_t* nitems,
                                                           int32_t* next_item) {
  __shared__ int64_t part[1024];
  const int64_t n = (int64_t)s.B * npairs;
  const int64_t per = (n + 1023) / 1024;
  const int64_t lo = threadIdx.x * per, hi = min(n, lo + per);
  // global tile order q: q = (npairs-1-p) * B + b
  int64_t cnt = 0;
  for (int64_t q = lo; q < hi; ++q) {
    const int b = (int)(q % s.B), p = npairs - 1 - (int)(q / s.B);
    cnt += (pair_kb_end(s, pos, b, p) + kSplitBlocks - 1) / kSplitBlocks;
  }
  part[threadIdx.x] = cnt;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    int64_t v = (int)threadIdx.x >= d ? part[threadIdx.x - d] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int64_t o = part[threadIdx.x] - cnt;
  for (int64_t q = lo; q < hi; ++q) {
    const int b = (int)(q % s.B), p = npairs - 1 - (int)(q / s.B);
    const int c = (pair_kb_end(s, pos, b, p) + kSplitBlocks - 1) / kSplitBlocks;
    for (int sp = 0; sp < c; ++sp) items[o++] = pack_item(b, p, sp);
  }
  if (threadIdx.x == 1023) *nitems = (int32_t)part[1023];
  if (threadIdx.x == 0) *next_item = 0;
}

__device__ __forceinline__ void item_range(const IndexTcArgs& a, int2 packed, int& b, int& p,
                                           int& sp, int& k0, int& k1) {
  sp = packed.y & 127;
  b = (packed.y >> 7) & 255;
  p = packed.x;
  k0 = sp * kSplitBlocks;
  k1 = min(k0 + kSplitBlocks, pair_kb_end(a.s, a.pos, b, p));
}

// Insert (cs, ci) into a list sorted by (score desc, id asc) when ci is larger
// than every id in the list (blocks are scanned in increasing order): its slot
// is the number of entries with score >= cs, and everything from there shifts
// down by one.  The caller checks cs > sc[last] first.  All steps are
// independent, so the update is short and has no serial chain.
__device__ __forceinline__ void list_insert_newest(float (&sc)[kCand], int (&id)[kCand], float cs,
                                                   int ci) {
  int k = 0;
#pragma unroll
  for (int j = 0; j < kCand; ++j) k += sc[j] >= cs ? 1 : 0;
#pragma unroll
  for (int j = kCand - 1; j > 0; --j) {
    sc[j] = j > k ? sc[j - 1] : (j == k ? cs : sc[j]);
    id[j] = j > k ? id[j - 1] : (j == k ? ci : id[j]);
  }
  if (k == 0) {
    sc[0] = cs;
    id[0] = ci;
  }
}

template <int DI>
__global__ void __launch_bounds__(kThreads, 1)
    index_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const IndexTcArgs a) {
  using C = IdxCfg<DI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;                              // [abuf][128 rows][DI]
  uint8_t* sB = smem + C::kSmemA;                  // [stage][256 keys][DI]
  Cand* sX = reinterpret_cast<Cand*>(sB + C::kSmemB);  // [kEpiLists][15][128 rows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sX) + C::kSmemX);
  uint64_t* full = bars;                          // kStages
  uint64_t* empty = full + kStages;               // kStages
  uint64_t* a_full = empty + kStages;             // 2
  uint64_t* a_empty = a_full + 2;                 // 2
  uint64_t* tm_full = a_empty + 2;                // kAccStages
  uint64_t* tm_empty = tm_full + kAccStages;      // kAccStages
  uint64_t* mma_done = tm_empty + kAccStages;     // 1
  uint64_t* it_full = mma_done + 1;               // kItemRing: an item id is published
  uint64_t* it_empty = it_full + kItemRing;       // kItemRing: every consumer has read it
  int* item_ring = reinterpret_cast<int*>(it_empty + kItemRing);  // kItemRing ids (-1: no more)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(item_ring + kItemRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_stop = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    *epi_stop = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kAccStages; ++i) {
      mbar_init(&tm_full[i], 1);
      mbar_init(&tm_empty[i], kEpiWarps / 2);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&it_full[i], 1);
      mbar_init(&it_empty[i], 1 + kEpiWarps);  // the MMA warp and every epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int T = a.s.T, G = a.s.G;
  const int nitems = *a.nitems;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      int stage = 0, abuf = 0;
      uint32_t sphase = 0, aphase = 0;
      int issued = 0, a_issued = 0;
      for (int ki = 0;; ++ki) {
        // take the next item and publish its id (-1 once none is left, or
        // after an abort) to the MMA warp and the epilogue
        const int slot = ki % kItemRing;
        if (ki >= kItemRing &&
            !mbar_wait(&it_empty[slot], ((ki / kItemRing) - 1) & 1, a.status, a.wait_polls)) {
          *abort_flag = 1;
          break;
        }
        int it = *abort_flag ? nitems : atomicAdd(a.next_item, 1);
        if (it >= nitems) it = -1;
        item_ring[slot] = it;
        mbar_arrive(&it_full[slot]);
        if (it < 0) break;
        int b, p, sp, k0, k1;
        item_range(a, a.items[it], b, p, sp, k0, k1);
        if (!mbar_wait(&a_empty[abuf], aphase ^ 1, a.status, a.wait_polls)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&a_full[abuf], C::kTileBytes);
        tma_load_2d(smem_u32(sA + abuf * C::kTileBytes), &tm_q, &a_full[abuf], 0,
                    (b * T) * G + p * kItemRows);
        ++a_issued;
        if (++abuf == 2) { abuf = 0; aphase ^= 1; }
        for (int kb = k0; kb < k1; kb += 2) {
          if (!mbar_wait(&empty[stage], sphase ^ 1, a.status, a.wait_polls)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          const uint32_t dst = smem_u32(sB + stage * C::kStageBytes);
          // the second block may lie past the item's range (odd count): its
          // scores are ignored; past the tensor's end the copy reads zeros
          int row0, row1;
          if (!a.s.bt) {
            row0 = (int)(b * a.cap + (int64_t)kb * kBlock);
            row1 = row0 + kBlock;
          } else {
            // paged: each block through the table; an entry outside the pool
            // (flagged) reads zeros from past the pool's end
            const int oob = (int)(a.s.cache_blocks() * kBlock);
            const int64_t p0 = cache_block(a.s, b, kb, a.status);
            const int64_t p1 = kb + 1 < k1 ? cache_block(a.s, b, kb + 1, a.status) : p0;
            row0 = p0 < 0 ? oob : (int)(p0 * kBlock);
            row1 = p1 < 0 ? oob : (int)(p1 * kBlock);
          }
          tma_load_2d(dst, &tm_k, &full[stage], 0, row0);
          tma_load_2d(dst + C::kBoxBytes, &tm_k, &full[stage], 0, row1);
          ++issued;
          if (++stage == kStages) { stage = 0; sphase ^= 1; }
        }
      }
      // No copy may still be landing in shared memory when the CTA exits: wait
      // (bounded) for the last load issued into each K_idx stage and each
      // Q_idx buffer.  Without an abort they were all consumed, and the waits
      // return at once; after one (a wait ran out anywhere in the CTA, maybe
      // after this loop ended) the consumers may have skipped them.
      {
        int n = issued < kStages ? issued : kStages;
        int st = stage;
        uint32_t ph = sphase;
        for (int k = 0; k < n; ++k) {
          if (st == 0) { st = kStages - 1; ph ^= 1; } else { --st; }
          mbar_wait(&full[st], ph, nullptr);
        }
        n = a_issued < 2 ? a_issued : 2;
        int ab = abuf;
        uint32_t aph = aphase;
        for (int k = 0; k < n; ++k) {
          if (ab == 0) { ab = 1; aph ^= 1; } else { --ab; }
          mbar_wait(&a_full[ab], aph, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // The whole warp runs the loop (waits and bookkeeping); one elected lane
    // issues the MMAs and commits.  Descriptors are formed once per buffer
    // and stepped by adding byte offsets / 16 to their start-address field.
    // Measured on the attention kernel's MMA warp: this halves the time to
    // issue a tile's MMAs against a loop run by lane 0 alone.
    {
      constexpr uint32_t idesc = idesc_bf16(128, kPairKeys, false, false);
      const uint64_t adesc0 = smem_desc(smem_u32(sA), 16, C::kSbo, C::kSwz);
      const uint64_t bdesc0 = smem_desc(smem_u32(sB), 16, C::kSbo, C::kSwz);
      int stage = 0, abuf = 0, ts = 0;
      uint32_t sphase = 0, aphase = 0, tphase = 0;
      for (int ki = 0;; ++ki) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // warp-uniform
        const int slot = ki % kItemRing;
        if (!__all_sync(0xffffffffu, mbar_wait(&it_full[slot], (ki / kItemRing) & 1, a.status, a.wait_polls))) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        // every lane's read of the slot is consumed (by the shuffle) before the
        // slot is handed back, so no read can still be pending when it is rewritten
        const int it = __shfl_sync(0xffffffffu, item_ring[slot], 0);
        if (lane == 0) mbar_arrive(&it_empty[slot]);
        if (it < 0) break;
        int b, p, sp, k0, k1;
        item_range(a, a.items[it], b, p, sp, k0, k1);
        if (!__all_sync(0xffffffffu, mbar_wait(&a_full[abuf], aphase, a.status, a.wait_polls))) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint64_t ad = adesc0 + (uint64_t)((abuf * C::kTileBytes) >> 4);
        bool ok = true;
        for (int kb = k0; kb < k1; kb += 2) {
          const bool okl = mbar_wait(&full[stage], sphase, a.status, a.wait_polls) &&
                           mbar_wait(&tm_empty[ts], tphase ^ 1, a.status, a.wait_polls);
          if (!__all_sync(0xffffffffu, okl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = bdesc0 + (uint64_t)((stage * C::kStageBytes) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < C::kKSteps; ++k)
              tc_mma_f16(tmem + ts * kPairKeys, ad + (uint64_t)(k * 2), bd + (uint64_t)(k * 2), idesc,
                         k > 0);
            tc_commit(&tm_full[ts]);
            tc_commit(&empty[stage]);
          }
          __syncwarp();
          if (++ts == kAccStages) { ts = 0; tphase ^= 1; }
          if (++stage == kStages) { stage = 0; sphase ^= 1; }
        }
        if (!ok) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        if (elect_one()) tc_commit(&a_empty[abuf]);
        __syncwarp();
        if (++abuf == 2) { abuf = 0; aphase ^= 1; }
      }
      // all MMAs issued by this warp complete before TMEM is released
      if (elect_one()) tc_commit(mma_done);
      __syncwarp();
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    // Four warpgroups (warps 2-17).  Warpgroups 0 and 1 read accumulator
    // stage 0, warpgroups 2 and 3 stage 1; within a stage, the even warpgroup
    // of the pair takes the first key block, the odd one the second.  Stages
    // alternate, so each warp has two stage-times per 128-score block.
    const int wg = (warp - 2) >> 2;     // 0..3
    const int my_ts = wg >> 1;          // accumulator stage this warpgroup reads
    const int half = wg & 1;            // which key block of the stage
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + my_ts * kPairKeys +
                               half * kBlock;
    uint32_t tphase = 0;
    int gstage = 0;                     // global stage count of this CTA at the item start
    // The 16 epilogue warps meet at named barriers per item, which have no
    // timeout; they stop together, on a shared stop word written before the
    // last barrier and read after it.
    bool stop = false;
    for (int ki = 0; !stop; ++ki) {
      // the 16 warps go on only together (a wait that ran out in one of them
      // stops all, at the same barrier)
      const int slot = ki % kItemRing;
      const bool okw =
          __all_sync(0xffffffffu, mbar_wait(&it_full[slot], (ki / kItemRing) & 1, a.status, a.wait_polls));
      // every lane's read of the slot is consumed (by the shuffle) before the
      // slot is handed back, so no read can still be pending when it is rewritten
      const int it = __shfl_sync(0xffffffffu, item_ring[slot], 0);
      if (lane == 0) mbar_arrive(&it_empty[slot]);
      if (!named_bar_and(1, 512, okw)) {
        stop = true;
        break;
      }
      if (it < 0) break;
      int b, p, sp, k0, k1;
      item_range(a, a.items[it], b, p, sp, k0, k1);
      const int local = p * kItemRows + r;  // row within sequence b
      const bool valid = local < T * G;
      const int qi = local / G, g = local - (local / G) * G;
      const int lb = valid ? (int)(((int64_t)a.pos.q_start[b] + qi) / kBlock) : 0;
      float sc[kCand];
      int id[kCand];
#pragma unroll
      for (int j = 0; j < kCand; ++j) {
        sc[j] = -INFINITY;
        id[j] = INT_MAX;
      }
      const int nst = (k1 - k0 + 1) >> 1;
      bool ok = true;
      // this warpgroup's stages of the item: global index == my_ts (mod 2)
      for (int q = ((my_ts - gstage) & 1); q < nst; q += 2) {
        if (!__all_sync(0xffffffffu, mbar_wait(&tm_full[my_ts], tphase, a.status, a.wait_polls))) { ok = false; break; }
        tphase ^= 1;
        tc_fence_after();
        // 16-column loads, two in flight per wait: small loads leave the
        // concurrently accumulating MMA more of tensor memory than larger
        // ones, and pairing them halves the round trips (measured: the stage
        // is read in about 500 instead of 700 cycles).  The load itself
        // reduces each lane's 16 scores to their maximum, so the block
        // max-pool costs no ALU work beyond combining eight partial maxima.
        float m = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          const float c0 = tmem_ld16_red<true>(lane_base + c * 16);
          const float c1 = tmem_ld16_red<true>(lane_base + c * 16 + 16);
          tmem_ld_wait();
          m = fmax3(m, c0, c1);
        }
        // the stage's scores are all read: the MMA may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tm_empty[my_ts]);
        const int blk = k0 + 2 * q + half;
        if (valid && blk < k1 && blk < lb && m > sc[kCand - 1]) list_insert_newest(sc, id, m, blk);
      }
      gstage += nst;
      // Merge of the four warpgroups' lists of each row, in one parallel
      // step: every list goes to shared memory, and each thread ranks its own
      // 15 candidates among all 60 (its position in its list plus, for each
      // other list, how many of its entries are better: a binary search, the
      // lists being sorted).  Ranks of real candidates are distinct (block ids
      // are), so the ranks below 15 fill the output once; empty entries rank
      // after every real one and fill the remaining slots with equal values.
      // Merging by serial insertion instead kept the epilogue from the next
      // item's accumulator stages for most of 30,000 cycles per item.
#pragma unroll
      for (int j = 0; j < kCand; ++j) sX[(wg * kCand + j) * kTileRows + r] = Cand{sc[j], id[j]};
      asm volatile("bar.sync 1, 512;" ::: "memory");
      if (valid && ok) {
        Cand* out = a.cand + ((((size_t)b * T + qi) * a.nsplit + sp) * G + g) * kCand;
        // own candidates are read back from shared memory, so that the loop
        // needs no run-time index into the register lists
#pragma unroll 1
        for (int j = 0; j < kCand; ++j) {
          const Cand own = sX[(wg * kCand + j) * kTileRows + r];
          const float cs = own.score;
          const int ci = own.id;
          int rank = j;
#pragma unroll 1
          for (int o = 1; o < kEpiLists; ++o) {
            const Cand* x = sX + (((wg + o) % kEpiLists) * kCand) * kTileRows + r;
            int lo = 0, hi = kCand;  // entries of list x better than (cs, ci): a prefix
#pragma unroll
            for (int step = 0; step < 4; ++step) {
              const int mid = min((lo + hi) >> 1, kCand - 1);  // read stays in the list
              const Cand c = x[mid * kTileRows];
              const bool better = c.score > cs || (c.score == cs && c.id < ci);
              if (lo < hi) {
                lo = better ? mid + 1 : lo;
                hi = better ? hi : mid;
              }
            }
            rank += lo;
          }
          if (rank < kCand) out[rank] = Cand{cs, ci};
        }
      }
      if (!ok || *abort_flag) *epi_stop = 1;
      asm volatile("bar.sync 1, 512;" ::: "memory");
      stop = *epi_stop != 0;
    }
    if (stop) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int index_tc_nsplit(int max_blocks) {
  const int n = (max_blocks - 1 + kSplitBlocks - 1) / kSplitBlocks;
  return n > 0 ? n : 1;
}

int index_tc_npairs(const Shape& s) {
  return (int)((s.T * (int64_t)s.G + kItemRows - 1) / kItemRows);
}

// scratch layout: [candidate lists][item count (256 B)][items]
size_t cand_bytes(const Shape& s) {
  const size_t c = (size_t)s.B * s.T * index_tc_nsplit(s.max_blocks) * s.G * kCand * sizeof(Cand);
  return (c + 255) / 256 * 256;
}

size_t items_cap(const Shape& s) {
  return (size_t)s.B * index_tc_npairs(s) * index_tc_nsplit(s.max_blocks);
}

template <int DI>
cudaError_t launch_index_tc_impl(const Shape& s, const Positions& pos, const uint16_t* q_idx,
                                 const uint16_t* k_idx, int32_t* sel, const Workspace& ws,
                                 cudaStream_t st) {
  using C = IdxCfg<DI>;
  const int64_t rows = (int64_t)s.B * s.T * s.G;
  const int64_t cap = (int64_t)s.max_blocks * kBlock;
  CUtensorMap tm_q, tm_k;
  {
    cuuint64_t dims[2] = {(cuuint64_t)DI, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)DI * 2};
    cuuint32_t box[2] = {(cuuint32_t)DI, (cuuint32_t)kTileRows};
    if (!encode_bf16_map(&tm_q, q_idx, 2, dims, strides, box,
                         DI == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)DI, (cuuint64_t)(s.cache_blocks() * kBlock)};
    cuuint64_t strides[1] = {(cuuint64_t)DI * 2};
    cuuint32_t box[2] = {(cuuint32_t)DI, (cuuint32_t)kBlock};
    if (!encode_bf16_map(&tm_k, k_idx, 2, dims, strides, box,
                         DI == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  char* base = reinterpret_cast<char*>(ws.cand);
  int32_t* nitems = reinterpret_cast<int32_t*>(base + cand_bytes(s));
  int2* items = reinterpret_cast<int2*>(nitems + 64);
  IndexTcArgs a;
  a.s = s;
  a.pos = pos;
  a.npairs = index_tc_npairs(s);
  a.nsplit = index_tc_nsplit(s.max_blocks);
  a.cap = cap;
  a.items = items;
  a.nitems = nitems;
  a.next_item = nitems + 1;
  a.cand = ws.cand;
  a.status = ws.status;
  a.wait_polls = debug_wait_polls();
  cudaError_t e = cudaFuncSetAttribute(index_tc_kernel<DI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const size_t maxitems = items_cap(s);
  const int grid = maxitems < (size_t)sm_count() ? (int)maxitems : sm_count();
  note_launches(2);
  index_items_kernel<<<1, 1024, 0, st>>>(s, pos, a.npairs, items, nitems, nitems + 1);
  index_tc_kernel<DI><<<grid, kThreads, C::kSmem, st>>>(tm_q, tm_k, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_topk_merge(s, pos, 0, s.T, kSplitBlocks, a.nsplit, ws.cand, sel, st);
}

}  // namespace

size_t tc_index_workspace_bytes(const Shape& s) {
  return cand_bytes(s) + 256 + items_cap(s) * sizeof(int2);
}

cudaError_t launch_index_tc(const Shape& s, const Positions& pos, const uint16_t* q_idx,
                            const uint16_t* k_idx, int32_t* sel, const Workspace& ws,
                            cudaStream_t st) {
  if (s.Di == 64) return launch_index_tc_impl<64>(s, pos, q_idx, k_idx, sel, ws, st);
  return launch_index_tc_impl<32>(s, pos, q_idx, k_idx, sel, ws, st);
}

}  // namespace msa
