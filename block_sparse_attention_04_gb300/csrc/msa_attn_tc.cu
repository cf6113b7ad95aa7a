// KV-outer sparse attention on tensor cores (prefill): step 4 of "MiniMax
// 模型迭代与竞品分析" section 2 (exact softmax over the selected blocks only),
// organised around the KV blocks, the "KV-outer" order that "MiniMax：Text-01 /
// M1 → M2.7 → M3" section 5 names for MSA's sparse kernel.
//
// A query-outer tile would hold one query's heads of one group (6 rows),
// far below the 128 rows a tcgen05 MMA wants.  So the selections are inverted:
// for every (sequence b, KV block kb, group g) the (query, slot) entries that
// chose it.  One tile = one such block x up to R entries, an entry's H/G heads
// padded to rpe = 8 (or 16) rows, i.e. at most 128 query-head rows against
// the block's 128 tokens.  One persistent CTA per SM runs two tile chains
// (tile t on chain t & 1), so one chain's S = Q K^T runs while the other
// chain's softmax works:
//   warp 0        TMA of Q tiles (8-head x D boxes, one per 8-row group)
//                 through a 3-deep ring: the Q copy is the longest latency
//   warp 1        TMA of K and V blocks of KV head g (block-major cache: 128
//                 rows of D bf16 at stride G*D) through 2-deep rings, one load
//                 per list
//   warp 2        tcgen05.mma, S(t) then P.V(t-1): S into TMEM, O = P V with P
//                 read from TMEM and V an MN-major smem operand
//   warps 3-10    row softmax, one warpgroup per chain (block-local max m, sum
//                 l; causal mask on the local block), P as bf16 written over S
//   warps 11-18   O as an unnormalised bf16 partial, one warpgroup per chain
// Each (query, head, slot) partial (O, m, l) is combined by a log-sum-exp
// merge into the bf16 output.
#include <climits>

#include "msa_device.cuh"
#include "msa_tc.h"
#include "msa_tma.h"

namespace msa {
namespace {

// warps: Q TMA, K/V TMA, MMA, 2 softmax warpgroups, 2 O-epilogue warpgroups
constexpr int kQWarp = 0, kKVWarp = 1, kMmaWarp = 2, kSoftWarp0 = 3, kEpiWarp0 = 11;
constexpr int kAttnThreads = 32 * 19;
constexpr int kPassRows = 8192;    // (sequence, query) rows per pass

struct AttnPass {
  Shape s;
  Positions pos;
  int t0, Tp;            // queries [t0, t0+Tp) of every sequence
  int nbl;               // key blocks per (sequence, group) in the list space
  int nlists;            // B * nbl * G
  int R;                 // entries per tile = 128 / rpe
  int rpe;               // tile rows per entry: H/G rounded up to 8 or 16
  const int32_t* sel;    // [B][T][G][16]
  int32_t* count;        // [nlists]
  int32_t* off;          // [nlists + 1]   entry offsets
  int32_t* tile_off;     // [nlists + 1]   tile offsets; tile_off[nlists] = total
  int32_t* entries;      // packed (i - t0) * 16 + slot
  int4* tile_desc;       // per tile: list, first entry, entries, kb | g << 15 | b << 18
  uint16_t* part_o;      // [B*Tp*H*16][D] bf16, O = sum 2^(s-m) v (unnormalised)
  float2* part_ml;       // [B*Tp*H*16] (m in log2 units, l)
  int* status;
  uint32_t wait_polls;   // poll cap of the pipeline waits (0: wall-clock bound only)
};

// Lists are ordered group-major, list (b, kb, g) at index (g*B + b)*nbl + kb:
// the tiles of one KV group are contiguous, so CTAs dealt nearby tiles all
// work on one group at a time.

__device__ __forceinline__ bool slot_valid(const AttnPass& a, int b, int i, int kb) {
  const int64_t t = (int64_t)a.pos.q_start[b] + i;
  return kb >= 0 && kb <= (int)(t / kBlock) && kb < a.s.max_blocks;
}

// ---- inverted lists -------------------------------------------------------
// The count and fill kernels give each CTA a contiguous range of the lists of
// one KV group (list_of is contiguous in (b, kb) for a fixed g).  The CTA
// reads every selection of its group in the pass and keeps the counts (or
// fill cursors) of its own lists in shared memory, so no global atomics are
// needed: with one global atomic per (query, group, slot) the two kernels
// were bound by atomic throughput (43 and 38 us per 8192-query pass at 128K).
constexpr int kCsrThreads = 512;
constexpr int kCsrMaxLists = 16384;  // shared-memory counters per CTA

struct CsrGrid {
  int per_group;   // CTAs per group
  int span;        // lists per CTA (the last CTA of a group may hold fewer)
};

inline CsrGrid csr_grid(const Shape& s, int nbl) {
  const int64_t lists_pg = (int64_t)s.B * nbl;
  int per = (sm_count() + s.G - 1) / s.G;
  const int64_t need = (lists_pg + kCsrMaxLists - 1) / kCsrMaxLists;
  if (per < need) per = (int)need;
  if (per > lists_pg) per = (int)(lists_pg > 0 ? lists_pg : 1);
  return CsrGrid{per, (int)((lists_pg + per - 1) / per)};
}

// This CTA's group and list range [lo, hi) within the group's B * nbl lists.
__device__ __forceinline__ void csr_cta_range(const AttnPass& a, int span, int per_group, int& g,
                                              int& lo, int& hi) {
  g = (int)blockIdx.x / per_group;
  const int c = (int)blockIdx.x % per_group;
  const int lists_pg = a.s.B * a.nbl;
  lo = min(lists_pg, c * span);
  hi = min(lists_pg, lo + span);
}

// One (sequence, query) row of group g per thread and step: its 16 slots are
// one 64-byte read, validated against the query's local block.
__global__ void __launch_bounds__(kCsrThreads) csr_count_kernel(AttnPass a, int span,
                                                                int per_group) {
  extern __shared__ int32_t s_cnt[];
  int g, lo, hi;
  csr_cta_range(a, span, per_group, g, lo, hi);
  const int nl = hi - lo;
  for (int k = threadIdx.x; k < nl; k += blockDim.x) s_cnt[k] = 0;
  __syncthreads();
  const int rows = a.s.B * a.Tp;
  const bool first = blockIdx.x % per_group == 0;  // one CTA per group flags bad ids
  for (int r = threadIdx.x; r < rows; r += blockDim.x) {
    const int b = r / a.Tp, i = a.t0 + r % a.Tp;
    const int4* sr = reinterpret_cast<const int4*>(
        a.sel + (((size_t)b * a.s.T + i) * a.s.G + g) * kTopk);
    const int64_t t = (int64_t)a.pos.q_start[b] + i;
    const int64_t lb = t / kBlock;
    const int lim = (int)(lb < a.s.max_blocks - 1 ? lb : a.s.max_blocks - 1);
    const int base = b * a.nbl - lo;
#pragma unroll
    for (int v = 0; v < kTopk / 4; ++v) {
      const int4 q4 = sr[v];
      const int ks[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kb = ks[u];
        if (kb < 0) continue;
        if (kb > lim) {
          if (first) flag_invalid(a.status);
          continue;
        }
        const int l = base + kb;
        if ((unsigned)l < (unsigned)nl) atomicAdd(&s_cnt[l], 1);
      }
    }
  }
  __syncthreads();
  int32_t* cnt = a.count + (size_t)g * a.s.B * a.nbl + lo;
  for (int k = threadIdx.x; k < nl; k += blockDim.x) cnt[k] = s_cnt[k];
}

// Exclusive scans of entry counts and of tile counts, one CTA of 1024 threads.
// Each thread owns a contiguous run of lists, read and written with 16-byte
// accesses where the run is aligned.
__global__ void __launch_bounds__(1024) csr_scan_kernel(AttnPass a) {
  __shared__ int64_t s_e[1024], s_t[1024];
  const int n = a.nlists;
  const int per = ((n + 1023) / 1024 + 3) & ~3;  // a multiple of 4
  const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
  int64_t se = 0, st = 0;
  int k = lo;
  for (; k + 4 <= hi; k += 4) {
    const int4 c = *reinterpret_cast<const int4*>(a.count + k);
    se += (int64_t)c.x + c.y + c.z + c.w;
    st += (c.x + a.R - 1) / a.R + (c.y + a.R - 1) / a.R + (c.z + a.R - 1) / a.R +
          (c.w + a.R - 1) / a.R;
  }
  for (; k < hi; ++k) {
    const int c = a.count[k];
    se += c;
    st += (c + a.R - 1) / a.R;
  }
  s_e[threadIdx.x] = se;
  s_t[threadIdx.x] = st;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    int64_t ve = 0, vt = 0;
    if ((int)threadIdx.x >= d) {
      ve = s_e[threadIdx.x - d];
      vt = s_t[threadIdx.x - d];
    }
    __syncthreads();
    s_e[threadIdx.x] += ve;
    s_t[threadIdx.x] += vt;
    __syncthreads();
  }
  int64_t oe = s_e[threadIdx.x] - se, ot = s_t[threadIdx.x] - st;
  k = lo;
  for (; k + 4 <= hi; k += 4) {
    const int4 c = *reinterpret_cast<const int4*>(a.count + k);
    int4 o, t;
    o.x = (int)oe; t.x = (int)ot; oe += c.x; ot += (c.x + a.R - 1) / a.R;
    o.y = (int)oe; t.y = (int)ot; oe += c.y; ot += (c.y + a.R - 1) / a.R;
    o.z = (int)oe; t.z = (int)ot; oe += c.z; ot += (c.z + a.R - 1) / a.R;
    o.w = (int)oe; t.w = (int)ot; oe += c.w; ot += (c.w + a.R - 1) / a.R;
    *reinterpret_cast<int4*>(a.off + k) = o;
    *reinterpret_cast<int4*>(a.tile_off + k) = t;
  }
  for (; k < hi; ++k) {
    const int c = a.count[k];
    a.off[k] = (int32_t)oe;
    a.tile_off[k] = (int32_t)ot;
    oe += c;
    ot += (c + a.R - 1) / a.R;
  }
  if (threadIdx.x == 1023) {
    a.off[n] = (int32_t)s_e[1023];
    a.tile_off[n] = (int32_t)s_t[1023];
  }
}

__global__ void __launch_bounds__(kCsrThreads) csr_fill_kernel(AttnPass a, int span,
                                                               int per_group) {
  extern __shared__ int32_t s_cur[];
  int g, lo, hi;
  csr_cta_range(a, span, per_group, g, lo, hi);
  const int nl = hi - lo;
  for (int k = threadIdx.x; k < nl; k += blockDim.x) s_cur[k] = 0;
  __syncthreads();
  const size_t l0 = (size_t)g * a.s.B * a.nbl + lo;  // global index of this CTA's first list
  const int rows = a.s.B * a.Tp;
  for (int r = threadIdx.x; r < rows; r += blockDim.x) {
    const int b = r / a.Tp, il = r % a.Tp;
    const int4* sr = reinterpret_cast<const int4*>(
        a.sel + (((size_t)b * a.s.T + a.t0 + il) * a.s.G + g) * kTopk);
    const int64_t t = (int64_t)a.pos.q_start[b] + a.t0 + il;
    const int64_t lb = t / kBlock;
    const int lim = (int)(lb < a.s.max_blocks - 1 ? lb : a.s.max_blocks - 1);
    const int base = b * a.nbl - lo;
#pragma unroll
    for (int v = 0; v < kTopk / 4; ++v) {
      const int4 q4 = sr[v];
      const int ks[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kb = ks[u];
        const int l = base + kb;
        if (kb < 0 || kb > lim || (unsigned)l >= (unsigned)nl) continue;
        const int p = atomicAdd(&s_cur[l], 1);
        a.entries[a.off[l0 + l] + p] = il * kTopk + v * 4 + u;
      }
    }
  }
  // tile table, thread per list: one 16-byte descriptor per tile, so the
  // attention kernel reads a tile's coordinates with a single load
  for (int k = threadIdx.x; k < nl; k += blockDim.x) {
    const size_t L = l0 + k;
    const int t0 = a.tile_off[L], t1 = a.tile_off[L + 1];
    if (t0 == t1) continue;
    const int kb = (lo + k) % a.nbl, b = (lo + k) / a.nbl;
    const int cnt = a.count[L], o = a.off[L];
    for (int t = t0; t < t1; ++t) {
      const int e0 = (t - t0) * a.R;
      a.tile_desc[t] = make_int4((int)L, o + e0, min(a.R, cnt - e0), kb | (g << 15) | (b << 18));
    }
  }
}

// ---- the attention tile kernel ---------------------------------------------
constexpr int kTileChunk = 4;   // consecutive tiles dealt to a CTA at a time

// Local tile i of this CTA -> its descriptor (see the chunked deal in
// attn_tc_kernel).
struct CtaTiles {
  const int4* all;
  __device__ __forceinline__ int4 operator[](int i) const {
    return all[((i / kTileChunk) * (int)gridDim.x + (int)blockIdx.x) * kTileChunk + i % kTileChunk];
  }
};
constexpr int kQStages = 3;   // Q tiles in flight (the Q copy is the longest latency)
constexpr int kKVStages = 2;  // K and V blocks in flight

template <int D>
struct AttnCfg {
  static constexpr int kHalf = 128 * 128;              // one [128 rows][64] bf16 SW128 box
  static constexpr int kNHalf = D / 64;                // 64-dim halves of a row
  static constexpr int kQGroup = kNHalf * 1024;        // one 8-row group of the Q tile
  static constexpr int kSmemQ = 16 * kQGroup;          // Q tile (128 rows)
  static constexpr int kSmemK = kNHalf * kHalf;        // one K (or V) block of one KV head
  static constexpr int kSmem = kQStages * kSmemQ + 2 * kKVStages * kSmemK + 256 + 1024;
  // two chains: S/P at [0,128) and [128,256), O at [256,384) and [384,512)
  static constexpr uint32_t kTmemCols = 512;
};

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnPass a) {
  using C = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;                                  // [kQStages] Q tiles
  uint8_t* sK = sQ + kQStages * C::kSmemQ;             // [kKVStages] K blocks
  uint8_t* sV = sK + kKVStages * C::kSmemK;            // [kKVStages] V blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kKVStages * C::kSmemK);
  uint64_t* q_full = bars;                        // kQStages
  uint64_t* q_empty = q_full + kQStages;          // kQStages
  uint64_t* k_full = q_empty + kQStages;          // kKVStages
  uint64_t* k_empty = k_full + kKVStages;
  uint64_t* v_full = k_empty + kKVStages;
  uint64_t* v_empty = v_full + kKVStages;
  uint64_t* s_full = v_empty + kKVStages;         // per chain: S of its tile is in TMEM
  uint64_t* p_full = s_full + 2;                  // per chain: P written over S
  uint64_t* o_full = p_full + 2;                  // per chain: O of its tile is in TMEM
  uint64_t* o_empty = o_full + 2;                 // per chain: O read out
  uint64_t* bar_fin = o_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < kKVStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(&s_full[c], 1);
      mbar_init(&p_full[c], 128);
      mbar_init(&o_full[c], 1);
      mbar_init(&o_empty[c], 128);
    }
    mbar_init(bar_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int H = a.s.H, hpg = H / a.s.G;
  const int rshift = a.rpe == 8 ? 3 : 4;  // tile row -> entry
  // This CTA's tiles: chunks of kTileChunk consecutive tiles (mostly of one
  // list, so the K/V block in shared memory is reused within a chunk), dealt
  // round-robin.  With group-major lists, all CTAs then work within a narrow
  // stretch of the tile order, i.e. on one KV group at a time, whose Q rows
  // and K/V blocks stay in L2; contiguous ranges per CTA had every CTA on a
  // different group, and each query's Q rows were fetched from DRAM for
  // most of its 16 blocks.
  const int ntiles = a.tile_off[a.nlists];
  const int nchunks = (ntiles + kTileChunk - 1) / kTileChunk;
  const int my_chunks =
      (int)blockIdx.x < nchunks ? (nchunks - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  int n = my_chunks * kTileChunk;                          // tiles of this CTA
  if (my_chunks > 0 && (nchunks - 1) % (int)gridDim.x == (int)blockIdx.x)
    n -= nchunks * kTileChunk - ntiles;                    // it holds the partial last chunk
  const CtaTiles desc{a.tile_desc};

  if (warp == kQWarp) {
    // ---------------------------------------------------- Q TMA (warp 0)
    // Q tiles through a kQStages ring: the Q of tile t is loaded once S of
    // tile t - kQStages is done, i.e. well before S of t is due.  Entry e
    // fills tile rows [e*rpe, e*rpe + rpe) (its hpg heads, then heads of the
    // next group or token, or zero fill past the end: rows the softmax and
    // epilogue skip), one box of 8 rows x D dims per lane.  L2 policy: Q rows
    // are read again for each block their query selected (evict last).
    const uint64_t pol_q = l2_policy_evict_last();
    const int bpe = a.rpe >> 3;                   // boxes per entry
    const int box_e = lane / bpe;                 // this lane's entry
    const int box_r = (lane % bpe) * 8;           // its first row within the entry
    int q_last[kQStages];                         // last tile loaded into each slot
#pragma unroll
    for (int i = 0; i < kQStages; ++i) q_last[i] = -1;
    for (int t = 0; t < n; ++t) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // warp-uniform
      const int4 d = desc[t];
      const int ne = d.z;
      int qrow = 0;
      if (box_e < ne) {
        const int il = a.entries[d.y + box_e] >> 4;
        qrow = (int)(((int64_t)(d.w >> 18) * a.s.T + a.t0 + il) * H + ((d.w >> 15) & 7) * hpg +
                     box_r);
      }
      const int qs = t % kQStages;
      const uint32_t u = (uint32_t)(t / kQStages);
      if (!__all_sync(0xffffffffu, mbar_wait(&q_empty[qs], (u & 1) ^ 1, a.status, a.wait_polls))) {
        *abort_flag = 1;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&q_full[qs], (uint32_t)(ne * a.rpe * D * 2));
      __syncwarp();
      if (box_e < ne)
        tma_load_3d_hint(smem_u32(sQ + qs * C::kSmemQ + ((box_e * a.rpe + box_r) >> 3) * C::kQGroup),
                         &tm_q, &q_full[qs], 0, qrow, 0, pol_q);
      q_last[qs] = t;
    }
    // no copy may still be landing in shared memory when the CTA exits (after
    // a timeout elsewhere the tiles were not all consumed): wait, bounded, for
    // the last load of each slot
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kQStages; ++i)
        if (q_last[i] >= 0) mbar_wait(&q_full[i], (uint32_t)(q_last[i] / kQStages) & 1, nullptr);
    }
  } else if (warp == kKVWarp) {
    // -------------------------------------------------- K/V TMA (warp 1)
    // One K and one V block per list change, through a kKVStages ring; a
    // buffer is refilled once the last tile of its previous list is through
    // S (K) or P.V (V).  L2 policy: evict first (used once, from smem).
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_first();
      int kv = -1, prev = -1;
      int k_last[kKVStages], v_last[kKVStages];   // last list loaded into each slot
#pragma unroll
      for (int i = 0; i < kKVStages; ++i) k_last[i] = v_last[i] = -1;
      for (int t = 0; t < n && !*abort_flag; ++t) {
        const int4 d = desc[t];
        if (d.x == prev) continue;
        prev = d.x;
        ++kv;
        const int ks = kv % kKVStages;
        const uint32_t w = (uint32_t)(kv / kKVStages);
        const int kb = d.w & 0x7FFF, g = (d.w >> 15) & 7, b = d.w >> 18;
        // through the block table when the caches are paged; an entry outside
        // the pool (flagged) reads zeros from past the pool's end
        const int64_t pb = cache_block(a.s, b, kb, a.status);
        const int row = (int)((pb < 0 ? a.s.cache_blocks() : pb) * kBlock);
        if (!mbar_wait(&k_empty[ks], (w & 1) ^ 1, a.status, a.wait_polls)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&k_full[ks], C::kSmemK);
#pragma unroll
        for (int h = 0; h < C::kNHalf; ++h)
          tma_load_3d_hint(smem_u32(sK + ks * C::kSmemK + h * C::kHalf), &tm_k, &k_full[ks], h * 64, g,
                           row, pol_kv);
        k_last[ks] = kv;
        if (!mbar_wait(&v_empty[ks], (w & 1) ^ 1, a.status, a.wait_polls)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&v_full[ks], C::kSmemK);
#pragma unroll
        for (int h = 0; h < C::kNHalf; ++h)
          tma_load_3d_hint(smem_u32(sV + ks * C::kSmemK + h * C::kHalf), &tm_v, &v_full[ks], h * 64, g,
                           row, pol_kv);
        v_last[ks] = kv;
      }
      // as for Q: no copy may still be landing when the CTA exits
#pragma unroll
      for (int i = 0; i < kKVStages; ++i) {
        if (k_last[i] >= 0) mbar_wait(&k_full[i], (uint32_t)(k_last[i] / kKVStages) & 1, nullptr);
        if (v_last[i] >= 0) mbar_wait(&v_full[i], (uint32_t)(v_last[i] / kKVStages) & 1, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------ MMA (warp 2)
    // Order S(0), S(1), P.V(0), S(2), P.V(1), ...: the S of one chain runs
    // while the other chain's softmax works.  Tile t uses chain c = t & 1:
    // S and P in TMEM columns [128c, 128c + 128), O in [256 + 128c, ...).
    // tcgen05.mma executes in issue order, so S(t + 2) cannot overwrite the P
    // that P.V(t), issued before it, still reads.
    // The whole warp runs the loop; one elected lane issues the MMAs and
    // commits, from descriptors formed once per ring and stepped by byte
    // offset / 16 (measured: half the issue time of a loop run by lane 0).
    {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
      const uint64_t qdesc0 = smem_desc(smem_u32(sQ), 16, C::kQGroup, kSwizzle128B);
      const uint64_t kdesc0 = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
      const uint64_t vdesc0 = smem_desc(smem_u32(sV), C::kHalf, 1024, kSwizzle128B);
      int kv = -1, prev = -1;
      int pv_ks = 0;
      uint32_t pv_w = 0;
      bool pv_last = false, pv_first = false;
      bool ok = true;
      // the lists of tiles t and t + 1, loaded two tiles ahead (a load takes
      // about as long as issuing a tile's MMAs)
      int l0 = n > 0 ? desc[0].x : -1, l1 = n > 1 ? desc[1].x : -1;
      for (int t = 0; t <= n && ok; ++t) {
        int ks = 0;
        uint32_t w = 0;
        bool last = false, first = false;
        const int lt = l0, ln = l1;
        l0 = l1;
        l1 = t + 2 < n ? desc[t + 2].x : -1;
        if (t < n) {
          // ---- S(t)
          first = lt != prev;  // K and V are waited for once per list
          if (first) { prev = lt; ++kv; }
          ks = kv % kKVStages;
          w = (uint32_t)(kv / kKVStages);
          last = (t + 1 == n) || ln != lt;
          const int c = t & 1, qs = t % kQStages;
          const bool okl =
              mbar_wait(&q_full[qs], (uint32_t)(t / kQStages) & 1, a.status, a.wait_polls) &&
              (!first || mbar_wait(&k_full[ks], w & 1, a.status, a.wait_polls));
          ok = __all_sync(0xffffffffu, okl);
          if (!ok) break;
          tc_fence_after();
          const uint64_t qd = qdesc0 + (uint64_t)((qs * C::kSmemQ) >> 4);
          const uint64_t kd = kdesc0 + (uint64_t)((ks * C::kSmemK) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k)  // 16 dims: (k & 3) * 32 bytes within a 64-dim half
              tc_mma_f16(tmem + c * 128, qd + (uint64_t)(((k >> 2) * 1024 + (k & 3) * 32) >> 4),
                         kd + (uint64_t)(((k >> 2) * C::kHalf + (k & 3) * 32) >> 4), idesc_s,
                         k > 0);
            tc_commit(&q_empty[qs]);
            tc_commit(&s_full[c]);
            if (last) tc_commit(&k_empty[ks]);
          }
          __syncwarp();
        }
        if (t >= 1) {
          // ---- P.V(t - 1)
          const int tp = t - 1, c = tp & 1;
          const uint32_t j = (uint32_t)(tp >> 1);
          const bool okl =
              mbar_wait(&p_full[c], j & 1, a.status, a.wait_polls) &&
              (!pv_first || mbar_wait(&v_full[pv_ks], pv_w & 1, a.status, a.wait_polls)) &&
              (j == 0 || mbar_wait(&o_empty[c], (j - 1) & 1, a.status, a.wait_polls));
          ok = __all_sync(0xffffffffu, okl);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd = vdesc0 + (uint64_t)((pv_ks * C::kSmemK) >> 4);
          // P (bf16, two per column) is in TMEM columns [128c, 128c + 64)
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc_mma_f16_ts(tmem + 256 + c * 128, tmem + c * 128 + k * 8,
                            vd + (uint64_t)((k * 2048) >> 4), idesc_o, k > 0);
            tc_commit(&o_full[c]);
            if (pv_last) tc_commit(&v_empty[pv_ks]);
          }
          __syncwarp();
        }
        pv_ks = ks;
        pv_w = w;
        pv_last = last;
        pv_first = first;
      }
      if (!ok && lane == 0) *abort_flag = 1;
      // all MMAs done before TMEM is released
      if (elect_one()) tc_commit(bar_fin);
      __syncwarp();
      mbar_wait(bar_fin, 0, nullptr);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------ softmax (2 warpgroups, one per chain)
    const int c = (warp - kSoftWarp0) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + c * 128;
    const float sl = a.s.scale * kLog2e;
    for (int t = c; t < n; t += 2) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // warp-uniform
      const int4 d = desc[t];
      const int kb = d.w & 0x7FFF, g = (d.w >> 15) & 7, b = d.w >> 18;
      const int e = r >> rshift, hh = r & (a.rpe - 1);
      const bool valid = e < d.z && hh < hpg;
      int il = 0, slot = 0;
      if (valid) {
        const int en = a.entries[d.y + e];
        il = en >> 4;
        slot = en & 15;
      }
      const int64_t tq = (int64_t)a.pos.q_start[b] + a.t0 + il;
      // tokens kb*128 + col with col > lim are masked (only in the local block)
      const int lim = (int)(tq - (int64_t)kb * kBlock);
      const bool masked = __any_sync(0xffffffffu, valid && lim < kBlock - 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[c], (uint32_t)(t >> 1) & 1, a.status, a.wait_polls))) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      // TMEM is read in 16-column loads, each waited before the next: small
      // loads leave the MMAs of the other chain more of tensor memory than
      // larger ones (measured).
      // pass 1: row maximum of the scaled scores: the maximum of the raw
      // scores, or their minimum when the scale is negative
      const bool neg = sl < 0.f;
      float mx = neg ? INFINITY : -INFINITY;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        if (masked) {
          uint32_t h[16];
          tmem_ld16(lane_base + cc * 16, h);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float x = __uint_as_float(h[k]);
            const bool in = cc * 16 + k <= lim;
            mx = neg ? fminf(mx, in ? x : INFINITY) : fmaxf(mx, in ? x : -INFINITY);
          }
        } else {
          // the load reduces the 16 scores itself
          if (neg) {
            const float r = tmem_ld16_red<false>(lane_base + cc * 16);
            tmem_ld_wait();
            mx = fminf(mx, r);
          } else {
            const float r = tmem_ld16_red<true>(lane_base + cc * 16);
            tmem_ld_wait();
            mx = fmaxf(mx, r);
          }
        }
      }
      const float m = mx * sl;
      // pass 2: P = 2^(s*scale*log2e - m) as bf16, two per column, written
      // over S in TMEM: the 32 scores of columns [32cc, 32cc+32) are read (two
      // loads) before columns [16cc, 16cc+16) are written, and those belong to
      // chunks already read; row sum
      float l0 = 0.f, l1 = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t wv[16];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t h[16];
          tmem_ld16(lane_base + cc * 32 + hf * 16, h);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int k = 2 * u;
            const int uu = hf * 8 + u;
            // 6 of 16 pairs on the FMA pipe, the rest on the MUFU unit
            constexpr unsigned kPolyPairs = 0x4925u;  // uu = 0, 2, 5, 8, 11, 14
            const bool poly = (kPolyPairs >> uu) & 1u;
            const float x0 = fmaf(__uint_as_float(h[k]), sl, -m);
            const float x1 = fmaf(__uint_as_float(h[k + 1]), sl, -m);
            float p0 = poly ? exp2_poly(x0) : ex2(x0);
            float p1 = poly ? exp2_poly(x1) : ex2(x1);
            if (masked) {
              p0 = cc * 32 + hf * 16 + k <= lim ? p0 : 0.f;
              p1 = cc * 32 + hf * 16 + k + 1 <= lim ? p1 : 0.f;
            }
            l0 += p0;
            l1 += p1;
            wv[uu] = pack_bf16(p0, p1);
          }
        }
        tmem_st16(lane_base + cc * 16, wv);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[c]);
      if (valid) {
        const size_t prow = (((size_t)b * a.Tp + il) * H + (size_t)g * hpg + hh) * kTopk + slot;
        __stcs(a.part_ml + prow, make_float2(m, l0 + l1));
      }
    }
  } else {
    // ------------------------------------ O epilogue (2 warpgroups, one per chain)
    // O = P.V (unnormalised) as a bf16 partial; the merge divides by the
    // combined sum.
    const int c = (warp - kEpiWarp0) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + 256 + c * 128;
    for (int t = c; t < n; t += 2) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // warp-uniform
      const int4 d = desc[t];
      const int g = (d.w >> 15) & 7, b = d.w >> 18;
      const int e = r >> rshift, hh = r & (a.rpe - 1);
      const bool valid = e < d.z && hh < hpg;
      size_t prow = 0;
      if (valid) {
        const int en = a.entries[d.y + e];
        prow = (((size_t)b * a.Tp + (en >> 4)) * H + (size_t)g * hpg + hh) * kTopk + (en & 15);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&o_full[c], (uint32_t)(t >> 1) & 1, a.status, a.wait_polls))) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      uint16_t* dst = a.part_o + prow * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 16; ++cc) {
        uint32_t h[16];
        tmem_ld16(lane_base + cc * 16, h);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int e8 = 0; e8 < 2; ++e8) {
            uint4 pk;
            pk.x = pack_bf16(__uint_as_float(h[e8 * 8 + 0]), __uint_as_float(h[e8 * 8 + 1]));
            pk.y = pack_bf16(__uint_as_float(h[e8 * 8 + 2]), __uint_as_float(h[e8 * 8 + 3]));
            pk.z = pack_bf16(__uint_as_float(h[e8 * 8 + 4]), __uint_as_float(h[e8 * 8 + 5]));
            pk.w = pack_bf16(__uint_as_float(h[e8 * 8 + 6]), __uint_as_float(h[e8 * 8 + 7]));
            __stcs(reinterpret_cast<uint4*>(dst + cc * 16 + e8 * 8), pk);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&o_empty[c]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---- merge: one warp per (sequence, query, head) ----------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_tc_merge_kernel(AttnPass a, uint16_t* __restrict__ out) {
  constexpr int PER = D / 32;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int H = a.s.H, hpg = H / a.s.G;
  if (gw >= (int64_t)a.s.B * a.Tp * H) return;
  const int h = (int)(gw % H);
  const int64_t r = gw / H;
  const int b = (int)(r / a.Tp), il = (int)(r % a.Tp);
  const int i = a.t0 + il, g = h / hpg;
  const size_t prow0 = (((size_t)b * a.Tp + il) * H + h) * kTopk;
  float m = -INFINITY, l = 0.f;
  if (lane < kTopk) {
    const int kb = a.sel[(((size_t)b * a.s.T + i) * a.s.G + g) * kTopk + lane];
    if (slot_valid(a, b, i, kb)) {
      const float2 ml = __ldcs(a.part_ml + prow0 + lane);
      m = ml.x;
      l = ml.y;
    }
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  // partial j holds O_j = sum p v with p = 2^(s - m_j): weight 2^(m_j - M),
  // normaliser sum_j 2^(m_j - M) l_j
  const float w = (m == -INFINITY) ? 0.f : ex2(m - M);
  float W = w * l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int j = 0; j < kTopk; ++j) {
    const float wj = __shfl_sync(0xffffffffu, w, j);
    if (wj == 0.f) continue;
    const uint16_t* src = a.part_o + (prow0 + j) * D + lane * PER;
    if constexpr (PER == 4) {
      const uint2 u = __ldcs(reinterpret_cast<const uint2*>(src));
      acc[0] += wj * bf16lo(u.x);
      acc[1] += wj * bf16hi(u.x);
      acc[2] += wj * bf16lo(u.y);
      acc[3] += wj * bf16hi(u.y);
    } else {
      const uint32_t u = __ldcs(reinterpret_cast<const unsigned int*>(src));
      acc[0] += wj * bf16lo(u);
      acc[1] += wj * bf16hi(u);
    }
  }
  uint16_t* dst = out + (((size_t)b * a.s.T + i) * H + h) * D + lane * PER;
  const float inv = 1.f / W;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
}

struct AttnLayout {
  size_t lists, entries, count_off, off_off, toff_off, ent_off, tl_off, po_off, pml_off, total;
};

AttnLayout attn_layout(const Shape& s) {
  AttnLayout L{};
  const int tp = pass_len(s);
  L.lists = (size_t)s.B * s.max_blocks * s.G;
  L.entries = (size_t)s.B * tp * s.G * kTopk;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t o = 0;
  L.count_off = o;  o += al(L.lists * 4);
  L.off_off = o;    o += al((L.lists + 1) * 4);
  L.toff_off = o;   o += al((L.lists + 1) * 4);
  L.ent_off = o;    o += al(L.entries * 4);
  L.tl_off = o;     o += al(L.entries * 16);
  const size_t prows = (size_t)s.B * tp * s.H * kTopk;
  L.po_off = o;     o += al(prows * s.D * 2);
  L.pml_off = o;    o += al(prows * 8);
  L.total = o;
  return L;
}

template <int D>
cudaError_t launch_attn_tc_impl(const Shape& s, const Positions& pos, const uint16_t* q,
                                const uint16_t* k, const uint16_t* v, const int32_t* sel,
                                uint16_t* out, const Workspace& ws, cudaStream_t st) {
  using C = AttnCfg<D>;
  const AttnLayout lay = attn_layout(s);
  char* base = ws.tc_base;
  const int hpg = s.H / s.G;
  const int rpe = hpg <= 8 ? 8 : 16;
  CUtensorMap tm_q, tm_k, tm_v;
  {
    // q as (64 dims, B*T*H rows, D/64 halves): one box = 8 rows (heads) x all
    // D dims, written half after half, i.e. one 8-row group of the Q tile
    cuuint64_t dims[3] = {64, (cuuint64_t)s.B * s.T * s.H, (cuuint64_t)(D / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, 8, (cuuint32_t)(D / 64)};
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
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  // one CTA per SM: all 512 TMEM columns and ~225 KiB of shared memory
  cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if ((e = cudaFuncSetAttribute(csr_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kCsrMaxLists * 4)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(csr_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kCsrMaxLists * 4)) != cudaSuccess)
    return e;
  const int grid = sm_count();
  const int tp_max = pass_len(s);
  for (int t0 = 0; t0 < s.T; t0 += tp_max) {
    AttnPass a;
    a.s = s;
    a.pos = pos;
    a.t0 = t0;
    a.Tp = min(tp_max, s.T - t0);
    const int max_lb = max_local_block(s, pos, t0, t0 + a.Tp);
    a.nbl = max_lb + 1;
    a.nlists = s.B * a.nbl * s.G;
    a.rpe = rpe;
    a.R = 128 / rpe;
    a.sel = sel;
    a.count = reinterpret_cast<int32_t*>(base + lay.count_off);
    a.off = reinterpret_cast<int32_t*>(base + lay.off_off);
    a.tile_off = reinterpret_cast<int32_t*>(base + lay.toff_off);
    a.entries = reinterpret_cast<int32_t*>(base + lay.ent_off);
    a.tile_desc = reinterpret_cast<int4*>(base + lay.tl_off);
    a.part_o = reinterpret_cast<uint16_t*>(base + lay.po_off);
    a.part_ml = reinterpret_cast<float2*>(base + lay.pml_off);
    a.status = ws.status;
    a.wait_polls = debug_wait_polls();
    const CsrGrid cg = csr_grid(s, a.nbl);
    const unsigned csr_ctas = (unsigned)(s.G * cg.per_group);
    const size_t csr_smem = (size_t)cg.span * 4;
    note_launches(4);
    csr_count_kernel<<<csr_ctas, kCsrThreads, csr_smem, st>>>(a, cg.span, cg.per_group);
    csr_scan_kernel<<<1, 1024, 0, st>>>(a);
    csr_fill_kernel<<<csr_ctas, kCsrThreads, csr_smem, st>>>(a, cg.span, cg.per_group);
    attn_tc_kernel<D><<<grid, kAttnThreads, C::kSmem, st>>>(tm_q, tm_k, tm_v, a);
    const int64_t warps = (int64_t)s.B * a.Tp * s.H;
    note_launches(1);
    attn_tc_merge_kernel<D><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(a, out);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

int pass_len(const Shape& s) {
  int tp = kPassRows / s.B;
  if (tp < 1) tp = 1;
  return tp < s.T ? tp : (s.T > 0 ? s.T : 1);
}

size_t tc_attn_workspace_bytes(const Shape& s) { return attn_layout(s).total; }

cudaError_t launch_attn_tc(const Shape& s, const Positions& pos, const uint16_t* q,
                           const uint16_t* k, const uint16_t* v, const int32_t* sel,
                           uint16_t* out, const Workspace& ws, cudaStream_t st) {
  if (s.D == 128) return launch_attn_tc_impl<128>(s, pos, q, k, v, sel, out, ws, st);
  return launch_attn_tc_impl<64>(s, pos, q, k, v, sel, out, ws, st);
}

}  // namespace msa
