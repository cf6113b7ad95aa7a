// Streaming kernels of libmsa: one query row at a time, any shape.  They are
// the decode path (T = 1 per sequence) and a correct path for every prefill.
//
//   index_stream  steps 1-2 of "MiniMax 模型迭代与竞品分析", section 2 (global
//                 index scoring over the causal context, 128-token max pooling)
//                 plus a per-split partial top-15 (step 3).  K_idx is streamed
//                 from HBM once per (query, split) for all G groups at once: a
//                 warp-level bf16 mma (16 keys x 8 groups x 16 dims) with fp32
//                 accumulation, block maxima kept in registers/shared memory.
//   topk_merge    step 3: merges the per-split lists, forces the local block
//                 in, sorts ids ascending, pads with -1.
//   attn_dec      step 4: a persistent CTA per SM; whole selected K/V blocks
//                 of one KV head arrive by TMA through a ring of shared-memory
//                 stages, and an online softmax over a part of a (query,
//                 group)'s selected blocks (scores of all heads of the group
//                 and P.V by mma) leaves one unnormalised partial per part.
//   attn_merge    combines the parts' partials of each (query, head)
//                 (log-sum-exp merge) into the bf16 output.
#include <cfloat>
#include <climits>

#include "msa_device.cuh"
#include "msa_tma.h"

namespace msa {
namespace {

constexpr int kIdxWarps = 8;
constexpr int kMaxBps = 256;  // key blocks per index split (shared array bound)
constexpr int kMaxSplits = 128;

__device__ __forceinline__ bool cand_better(float s1, int i1, float s2, int i2) {
  return s1 > s2 || (s1 == s2 && i1 < i2);
}

__device__ __forceinline__ void warp_argbest(float& s, int& id, int& owner) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    int i2 = __shfl_xor_sync(0xffffffffu, id, o);
    int w2 = __shfl_xor_sync(0xffffffffu, owner, o);
    if (cand_better(s2, i2, s, id)) {
      s = s2;
      id = i2;
      owner = w2;
    }
  }
}

// ---------------------------------------------------------------------------
// index_stream: grid (nsplit, rows); 256 threads.  Row r of the pass is query
// i = t0 + r % Tp of sequence b = r / Tp.
template <int DI>
__global__ void __launch_bounds__(kIdxWarps * 32) index_stream_kernel(
    Shape s, Positions pos, int T, int t0, int Tp, int bps, int nsplit,
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx,
    Cand* __restrict__ cand, int* __restrict__ status) {
  constexpr int NJ = DI / 16;  // mma k-steps per key row
  constexpr int NU = DI / 32;  // 16-byte loads per key row and thread
  __shared__ float pooled[kMaxBps][8];

  const int split = blockIdx.x;
  const int row = blockIdx.y;
  const int b = row / Tp, i = t0 + row % Tp;
  const int64_t t = (int64_t)pos.q_start[b] + i;
  const int lb = (int)(t / kBlock);
  const int blk0 = split * bps;
  if (blk0 >= lb) return;  // the merge reads only the valid splits
  const int blk1 = min(blk0 + bps, lb);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int G = s.G;

  // B fragments: q_idx^T (dims x groups); column n = gq is group gq.
  uint32_t bq[NJ][2];
  {
    const uint16_t* qr = q_idx + ((size_t)(b * T + i) * G + (gq < G ? gq : 0)) * DI;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int base = (j >> 1) * 32 + 8 * tq + (j & 1) * 4;
      uint32_t lo = *reinterpret_cast<const uint32_t*>(qr + base);
      uint32_t hi = *reinterpret_cast<const uint32_t*>(qr + base + 2);
      bq[j][0] = gq < G ? lo : 0u;
      bq[j][1] = gq < G ? hi : 0u;
    }
  }

  // This warp's blocks are blk0 + warp + k * kIdxWarps, streamed in steps of
  // 16 key rows (8 steps per block).  The loads of step it + 1 are issued
  // before the MMAs of step it, so each warp keeps two steps in flight
  // (measured 4 % faster than one on the 64 x 256K decode batch; a two-step
  // lookahead spilled registers and was slower).
  constexpr int SPB = kBlock / 16;  // steps per block
  const int nbw = (blk1 - blk0 - warp + kIdxWarps - 1) / kIdxWarps;
  const int n = nbw > 0 ? nbw * SPB : 0;
  uint4 C0[NU], C1[NU];  // rows gq and gq + 8 of the current step
  // Row gq of the k-th block of this warp, resolved once per block (a
  // block-table entry outside the pool is flagged and block 0 read instead).
  const uint16_t* lrow = k_idx;
#define MSA_IDX_BLOCK(K)                                                                  \
  do {                                                                                    \
    const int64_t pb_ = cache_block(s, b, blk0 + warp + (K) * kIdxWarps, status);         \
    lrow = k_idx + ((size_t)(pb_ < 0 ? 0 : pb_) * kBlock + gq) * DI;                      \
  } while (0)
#define MSA_IDX_LOAD(STEP, X0, X1)                                                        \
  do {                                                                                    \
    const uint16_t* r_ = lrow + (STEP) * 16 * DI;                                         \
    _Pragma("unroll") for (int u_ = 0; u_ < NU; ++u_) {                                   \
      X0[u_] = ldg_stream(r_ + (tq + 4 * u_) * 8);                                        \
      X1[u_] = ldg_stream(r_ + 8 * DI + (tq + 4 * u_) * 8);                               \
    }                                                                                     \
  } while (0)
  if (n > 0) {
    MSA_IDX_BLOCK(0);
    MSA_IDX_LOAD(0, C0, C1);
  }
  float m0 = -INFINITY, m1 = -INFINITY;
  for (int it = 0; it < n; ++it) {
    uint4 N0[NU], N1[NU];
    if (it + 1 < n) {
      if ((it + 1) % SPB == 0) MSA_IDX_BLOCK((it + 1) / SPB);
      MSA_IDX_LOAD((it + 1) % SPB, N0, N1);
    } else {
#pragma unroll
      for (int u = 0; u < NU; ++u) N0[u] = N1[u] = make_uint4(0, 0, 0, 0);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int u = j >> 1;
      const bool e = j & 1;
      mma_bf16_16816(acc, e ? C0[u].z : C0[u].x, e ? C1[u].z : C1[u].x, e ? C0[u].w : C0[u].y,
                     e ? C1[u].w : C1[u].y, bq[j][0], bq[j][1]);
    }
    m0 = fmax3(m0, acc[0], acc[2]);
    m1 = fmax3(m1, acc[1], acc[3]);
    if (it % SPB == SPB - 1) {  // the block is complete: pool over the 8 row groups
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      }
      const int blk = blk0 + warp + (it / SPB) * kIdxWarps;
      if (gq == 0) {
        pooled[blk - blk0][2 * tq] = m0;
        pooled[blk - blk0][2 * tq + 1] = m1;
      }
      m0 = -INFINITY;
      m1 = -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      C0[u] = N0[u];
      C1[u] = N1[u];
    }
  }
#undef MSA_IDX_LOAD
#undef MSA_IDX_BLOCK
  __syncthreads();

  // Partial top-15 of this split, one warp per group, best first.
  const int nblk = blk1 - blk0;
  Cand* out = cand + ((size_t)row * nsplit + split) * G * kCand;
  for (int g = warp; g < G; g += kIdxWarps) {
    float last_s = INFINITY;
    int last_id = -1;
    for (int r = 0; r < kCand; ++r) {
      float bs = -INFINITY;
      int bid = INT_MAX, owner = 0;
      for (int c = lane; c < nblk; c += 32) {
        const float sc = pooled[c][g];
        const int id = blk0 + c;
        const bool eligible = sc < last_s || (sc == last_s && id > last_id);
        if (eligible && cand_better(sc, id, bs, bid)) {
          bs = sc;
          bid = id;
        }
      }
      warp_argbest(bs, bid, owner);
      if (lane == 0) out[g * kCand + r] = Cand{bs, bid};
      last_s = bs;
      last_id = bid;
    }
  }
}

// ---------------------------------------------------------------------------
// topk_merge: one warp per (pass row, group).
__global__ void __launch_bounds__(256) topk_merge_kernel(
    Shape s, Positions pos, int T, int t0, int Tp, int bps, int nsplit, int nrows,
    const Cand* __restrict__ cand, int32_t* __restrict__ sel) {
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= nrows * s.G) return;
  const int row = gw / s.G, g = gw % s.G;
  const int b = row / Tp, i = t0 + row % Tp;
  const int64_t t = (int64_t)pos.q_start[b] + i;
  const int lb = (int)(t / kBlock);
  const int nvalid = (lb + bps - 1) / bps;

  const Cand* base = cand + (size_t)row * nsplit * s.G * kCand + (size_t)g * kCand;
  const size_t lstride = (size_t)s.G * kCand;  // between the lists of consecutive splits
  int my_id = -1;
  if (nvalid == 1) {
    // one list: already the ranked top-15 of every candidate block
    if (lane < kCand) {
      const Cand c = base[lane];
      my_id = (c.id == INT_MAX || lane >= lb) ? -1 : c.id;
    }
  } else if (nvalid <= 32) {
    // lane l holds split l's sorted list in registers; the winner of each
    // round shifts its list by one
    float ls[kCand];
    int li[kCand];
#pragma unroll
    for (int k = 0; k < kCand; ++k) {
      Cand c = Cand{-INFINITY, INT_MAX};
      if (lane < nvalid) c = base[(size_t)lane * lstride + k];
      ls[k] = c.score;
      li[k] = c.id;
    }
    for (int r = 0; r < kCand; ++r) {
      float bs = ls[0];
      int bid = li[0], owner = lane;
      warp_argbest(bs, bid, owner);
      if (owner == lane) {
#pragma unroll
        for (int k = 0; k < kCand - 1; ++k) {
          ls[k] = ls[k + 1];
          li[k] = li[k + 1];
        }
        ls[kCand - 1] = -INFINITY;
        li[kCand - 1] = INT_MAX;
      }
      if (lane == r) my_id = (bid == INT_MAX || r >= lb) ? -1 : bid;
    }
  } else {
    // lane owns splits lane, lane+32, lane+64, lane+96; cursors into each list
    int cur[4] = {0, 0, 0, 0};
    for (int r = 0; r < kCand; ++r) {
      float bs = -INFINITY;
      int bid = INT_MAX, bk = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int sp = lane + 32 * k;
        if (sp < nvalid && cur[k] < kCand) {
          Cand c = base[(size_t)sp * lstride + cur[k]];
          if (cand_better(c.score, c.id, bs, bid)) {
            bs = c.score;
            bid = c.id;
            bk = k;
          }
        }
      }
      int owner = lane * 4 + bk;
      warp_argbest(bs, bid, owner);
      if ((owner >> 2) == lane) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k == (owner & 3)) ++cur[k];
      }
      if (lane == r) my_id = (bid == INT_MAX || r >= lb) ? -1 : bid;
    }
  }
  if (lane == kCand) my_id = lb;
  // ascending order, -1 padding last
  const int key = (lane < kTopk && my_id >= 0) ? my_id : INT_MAX;
  int rank = 0;
  for (int j = 0; j < kTopk; ++j) {
    const int kj = __shfl_sync(0xffffffffu, key, j);
    rank += (kj < key) || (kj == key && j < lane);
  }
  if (lane < kTopk) sel[((size_t)(b * T + i) * s.G + g) * kTopk + rank] = (key == INT_MAX) ? -1 : key;
}

// ---------------------------------------------------------------------------
// attn_dec: a persistent CTA per SM walks work items (pass row, group, part);
// a part is spp = 16 / nparts consecutive selection slots.  Warp 4 (one lane)
// reads the part's selected ids, resolves each to its cache block and copies
// the block's K and V (128 tokens x D of one KV head, two 3-D TMA boxes of 64
// dims each) into a ring of stages, and the group's query rows into one of
// two query buffers by a bulk copy, running ahead of the compute by the depth
// of the ring.  Warps 0-3 run an online softmax over the part's blocks:
// S^T = K Q^T (tokens x heads) and O^T += V^T P^T with mma.sync, operands
// read from the 128-byte-swizzled stages with ldmatrix; then one unnormalised
// partial (O relative to the running max m, and m, l) per (row, head, part).
struct DecArgs {
  Shape s;
  Positions pos;
  int T, t0, Tp, nparts, spp, nitems;
  const uint16_t* q;
  const int32_t* sel;
  float* part_o;
  float* part_ml;
  int* status;
  uint32_t wait_polls;
};

constexpr int kDecConsumers = 128;          // warps 0-3
constexpr int kDecThreads = kDecConsumers + 32;

template <int D, int NTH>
struct DecCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kBox = 64 * kBlock * 2;                // one 64-dim box, 16 KiB
  static constexpr int kStageBytes = 2 * kHalves * kBox;      // K boxes, then V boxes
  static constexpr int kStages = D == 128 ? 3 : 6;            // 192 KiB of blocks in flight
  static constexpr int NH = NTH * 8;
  static constexpr int PSTR = kBlock + 8;                     // padded P row (elements)
  static constexpr int kQBytes = NH * D * 2;
  static constexpr int kQBufs = 4;                            // query buffers (items ahead)
  static constexpr int kStagesOff = 0;
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kPOff = kQOff + kQBufs * kQBytes;
  static constexpr int kRedOff = kPOff + NH * PSTR * 2;       // [2][4][NH] float
  static constexpr int kLsumOff = kRedOff + 2 * 4 * NH * 4;   // [2][4][NH] float
  static constexpr int kMetaOff = kLsumOff + 2 * 4 * NH * 4;  // [kStages] int
  static constexpr int kBarOff = (kMetaOff + kStages * 4 + 7) / 8 * 8;
  static constexpr int kBytes = kBarOff + (2 * kStages + 2 * kQBufs) * 8;
  static constexpr int kSmem = kBytes + 1024;                 // base alignment slack
};

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a box written
// with the 128-byte swizzle (rows of 128 bytes, chunk index xor row % 8).
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int D, int NTH>
__global__ void __launch_bounds__(kDecThreads, 1) attn_dec_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ DecArgs a) {
  using C = DecCfg<D, NTH>;
  constexpr int NJ = D / 16;     // k-steps of the score mma
  constexpr int MGV = D / 64;    // 16-dim groups of O per warp
  constexpr int NH = C::NH;
  constexpr int S = C::kStages;
  constexpr int NQ = C::kQBufs;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint16_t* qbuf = reinterpret_cast<uint16_t*>(sm + C::kQOff);
  uint16_t* ps = reinterpret_cast<uint16_t*>(sm + C::kPOff);
  float* red = reinterpret_cast<float*>(sm + C::kRedOff);
  float* lsum = reinterpret_cast<float*>(sm + C::kLsumOff);
  int* meta_kb = reinterpret_cast<int*>(sm + C::kMetaOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
  uint64_t* empty = full + S;
  uint64_t* q_full = empty + S;
  uint64_t* q_empty = q_full + NQ;

  const Shape& s = a.s;
  const int H = s.H, G = s.G, hpg = H / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 4);
    }
    fence_mbar_init();
  }
  // query rows past the group's heads stay zero (their columns are computed
  // and never written)
  for (int e = threadIdx.x; e < NQ * NH * D / 2; e += blockDim.x) {
    const int r = (e * 2 / D) % NH;
    if (r >= hpg) reinterpret_cast<uint32_t*>(qbuf)[e] = 0u;
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const uint32_t qbytes = (uint32_t)(hpg * D * 2);
      int n = 0, k = 0, nq = 0;   // stages armed, items begun, query copies issued
      bool ok = true;
      for (int item = blockIdx.x; item < a.nitems && ok; item += gridDim.x, ++k) {
        const int unit = item / a.nparts, part = item % a.nparts;
        const int row = unit / G, g = unit % G;
        const int b = row / a.Tp, i = a.t0 + row % a.Tp;
        const int64_t t = (int64_t)a.pos.q_start[b] + i;
        const int lb = (int)(t / kBlock);
        const int qs = k % NQ;
        if (k >= NQ && !mbar_wait(&q_empty[qs], ((k / NQ) - 1) & 1, a.status, a.wait_polls)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&q_full[qs], qbytes);
        bulk_load(smem_u32(qbuf + qs * NH * D),
                  a.q + ((size_t)(b * a.T + i) * H + (size_t)g * hpg) * D, qbytes, &q_full[qs]);
        ++nq;
        const int32_t* srow = a.sel + ((size_t)(b * a.T + i) * G + g) * kTopk + part * a.spp;
        for (int j = 0; j < a.spp; ++j, ++n) {
          int kb = srow[j];
          if (kb > lb || kb >= s.max_blocks) {
            flag_invalid(a.status);
            kb = -1;
          }
          int64_t pb = -1;
          if (kb >= 0) {
            pb = cache_block(s, b, kb, a.status);
            if (pb < 0) kb = -1;
          }
          const int st = n % S;
          if (n >= S && !mbar_wait(&empty[st], ((n / S) - 1) & 1, a.status, a.wait_polls)) {
            ok = false;
            break;
          }
          meta_kb[st] = kb;
          if (kb < 0) {
            mbar_arrive(&full[st]);
            continue;
          }
          mbar_arrive_expect_tx(&full[st], C::kStageBytes);
          const uint32_t kdst = smem_u32(sm + C::kStagesOff + st * C::kStageBytes);
          const uint32_t vdst = kdst + C::kHalves * C::kBox;
          const int z = (int)(pb * kBlock);
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h) {
            tma_load_3d_hint(kdst + h * C::kBox, &tm_k, &full[st], h * 64, g, z, pol);
            tma_load_3d_hint(vdst + h * C::kBox, &tm_v, &full[st], h * 64, g, z, pol);
          }
        }
      }
      // Wait (wall clock only) for the last copies of every buffer, so that
      // none lands after the CTA has exited, also when the consumers have
      // given up or this lane stopped issuing after a wait ran out.
      for (int m = n - 1; m >= 0 && m >= n - S; --m) mbar_wait(&full[m % S], (m / S) & 1, nullptr);
      for (int m = nq - 1; m >= 0 && m >= nq - NQ; --m)
        mbar_wait(&q_full[m % NQ], (m / NQ) & 1, nullptr);
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gq = lane >> 2, tq = lane & 3;
  const float qk_scale = s.scale * kLog2e;
  int n = 0, vb = 0, k = 0;
  for (int item = blockIdx.x; item < a.nitems; item += gridDim.x, ++k) {
    const int unit = item / a.nparts, part = item % a.nparts;
    const int row = unit / G, g = unit % G;
    const int b = row / a.Tp, i = a.t0 + row % a.Tp;
    const int64_t t = (int64_t)a.pos.q_start[b] + i;
    const int lb = (int)(t / kBlock);
    const int qs = k % NQ;

    bool ok = mbar_wait(&q_full[qs], (k / NQ) & 1, a.status, a.wait_polls);
    if (!named_bar_and(1, kDecConsumers, ok)) return;
    // Q^T fragments (dims x heads) of this item
    uint32_t bq[NTH][NJ][2];
    {
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qbuf + qs * NH * D);
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int w0 = ((nt * 8 + gq) * D + j * 16 + 2 * tq) / 2;
          bq[nt][j][0] = q32[w0];
          bq[nt][j][1] = q32[w0 + 4];
        }
    }

    float o[MGV][NTH][4];
    float m_run[NTH][2], l_w[NTH][2];
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m_run[nt][e] = -INFINITY;
        l_w[nt][e] = 0.f;
      }
#pragma unroll
    for (int mg = 0; mg < MGV; ++mg)
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[mg][nt][c] = 0.f;

    for (int j = 0; j < a.spp; ++j, ++n) {
      const int st = n % S;
      ok = mbar_wait(&full[st], (n / S) & 1, a.status, a.wait_polls);
      if (!named_bar_and(1, kDecConsumers, ok)) return;
      const int kb = meta_kb[st];
      if (kb >= 0) {
        const uint32_t kbase = smem_u32(sm + C::kStagesOff + st * C::kStageBytes);
        const uint32_t vbase = kbase + C::kHalves * C::kBox;
        // scores S^T[token][head] of this warp's 32 tokens
        float sc[2][NTH][4];
#pragma unroll
        for (int mg = 0; mg < 2; ++mg) {
          const int tok = warp * 32 + mg * 16 + (lane & 15);
#pragma unroll
          for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[mg][nt][c] = 0.f;
#pragma unroll
          for (int jj = 0; jj < NJ; ++jj) {
            uint32_t ka[4];
            ldmatrix_x4(ka, kbase + (jj >> 2) * C::kBox +
                                swz128(tok, (jj & 3) * 2 + (lane >> 4)));
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt)
              mma_bf16_16816(sc[mg][nt], ka[0], ka[1], ka[2], ka[3], bq[nt][jj][0],
                             bq[nt][jj][1]);
          }
          const int64_t tok0 = (int64_t)kb * kBlock + warp * 32 + mg * 16 + gq;
#pragma unroll
          for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              sc[mg][nt][c] = (kb < lb || tok0 + (c >= 2 ? 8 : 0) <= t)
                                  ? sc[mg][nt][c] * qk_scale
                                  : -INFINITY;
        }
        // block max per head over the four warps, new running max
        float* rd = red + (vb & 1) * 4 * NH;
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float m = fmaxf(fmaxf(sc[0][nt][e], sc[0][nt][e + 2]),
                            fmaxf(sc[1][nt][e], sc[1][nt][e + 2]));
#pragma unroll
            for (int off = 4; off < 32; off <<= 1)
              m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (gq == 0) rd[warp * NH + nt * 8 + 2 * tq + e] = m;
          }
        named_bar_sync(1, kDecConsumers);
        float alpha[NTH][2];
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = nt * 8 + 2 * tq + e;
            const float bm = fmaxf(fmaxf(rd[h], rd[NH + h]), fmaxf(rd[2 * NH + h], rd[3 * NH + h]));
            const float mn = fmaxf(m_run[nt][e], bm);
            alpha[nt][e] = ex2(m_run[nt][e] - mn);
            m_run[nt][e] = mn;
          }
        // p = 2^(s - m) -> bf16 P[head][token]; this warp's row sums
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = nt * 8 + 2 * tq + e;
            float sum = 0.f;
#pragma unroll
            for (int mg = 0; mg < 2; ++mg)
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const float p = ex2(sc[mg][nt][e + 2 * rr] - m_run[nt][e]);
                sum += p;
                ps[h * C::PSTR + warp * 32 + mg * 16 + gq + 8 * rr] =
                    (uint16_t)f32_to_bf16_rne(p);
              }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            l_w[nt][e] = l_w[nt][e] * alpha[nt][e] + sum;
          }
#pragma unroll
        for (int mg = 0; mg < MGV; ++mg)
#pragma unroll
          for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[mg][nt][c] *= alpha[nt][c & 1];
        named_bar_sync(1, kDecConsumers);
        // O^T[dim][head] += V^T P^T; warp w owns dims [w*D/4, (w+1)*D/4)
        const uint32_t* p32 = reinterpret_cast<const uint32_t*>(ps);
#pragma unroll
        for (int ks = 0; ks < kBlock / 16; ++ks) {
#pragma unroll
          for (int mg = 0; mg < MGV; ++mg) {
            const int mi = lane >> 3;
            const int tok = ks * 16 + (lane & 7) + ((mi & 2) ? 8 : 0);
            const int dim = warp * (D / 4) + mg * 16 + ((mi & 1) ? 8 : 0);
            uint32_t va[4];
            ldmatrix_x4_trans(va, vbase + (dim >> 6) * C::kBox + swz128(tok, (dim & 63) >> 3));
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) {
              const int h = nt * 8 + gq;
              const uint32_t b0 = p32[(h * C::PSTR) / 2 + ks * 8 + tq];
              const uint32_t b1 = p32[(h * C::PSTR) / 2 + ks * 8 + 4 + tq];
              mma_bf16_16816(o[mg][nt], va[0], va[1], va[2], va[3], b0, b1);
            }
          }
        }
        ++vb;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // The query buffer goes back only now: the score MMAs have consumed the
    // fragments, so no load of them can still be outstanding when the next
    // copy overwrites the buffer.
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[qs]);

    // the item's partials: O relative to m, and (m, l) per head
    float* ls = lsum + (k & 1) * 4 * NH;
    if (gq == 0) {
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) ls[warp * NH + nt * 8 + 2 * tq + e] = l_w[nt][e];
    }
    named_bar_sync(1, kDecConsumers);
    const size_t hbase = ((size_t)row * H + (size_t)g * hpg) * a.nparts + part;
#pragma unroll
    for (int mg = 0; mg < MGV; ++mg)
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int h = nt * 8 + 2 * tq + (c & 1);
          const int dim = warp * (D / 4) + mg * 16 + gq + (c >= 2 ? 8 : 0);
          if (h < hpg) a.part_o[(hbase + (size_t)h * a.nparts) * D + dim] = o[mg][nt][c];
        }
    if (warp == 0 && gq == 0) {
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = nt * 8 + 2 * tq + e;
          if (h < hpg) {
            const float l = ls[h] + ls[NH + h] + ls[2 * NH + h] + ls[3 * NH + h];
            a.part_ml[(hbase + (size_t)h * a.nparts) * 2 + 0] = m_run[nt][e];
            a.part_ml[(hbase + (size_t)h * a.nparts) * 2 + 1] = l;
          }
        }
    }
  }
}

// ---------------------------------------------------------------------------
// attn_merge: one warp per (pass row, head), over its nparts partials.
// DENSE: fold into the dense accumulators instead (one chunk of msa_dense_attn).
template <int D, bool DENSE>
__global__ void __launch_bounds__(256) attn_merge_kernel(
    Shape s, int T, int t0, int Tp, int nrows, int nparts, const float* __restrict__ part_o,
    const float* __restrict__ part_ml, uint16_t* __restrict__ out, DenseStep ds) {
  constexpr int PER = D / 32;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= nrows * s.H) return;
  const int row = gw / s.H, h = gw % s.H;
  const int b = row / Tp, i = t0 + row % Tp;
  const size_t base = ((size_t)row * s.H + h) * nparts;
  float m = -INFINITY, l = 0.f;
  if (lane < nparts) {
    m = part_ml[(base + lane) * 2];
    l = part_ml[(base + lane) * 2 + 1];
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w = (m == -INFINITY) ? 0.f : ex2(m - M);
  float L = w * l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int j = 0; j < nparts; ++j) {
    const float wj = __shfl_sync(0xffffffffu, w, j);
    if (wj == 0.f) continue;
    const float* src = part_o + (base + j) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += wj * src[e];
  }
  uint16_t* dst = out + ((size_t)(b * T + i) * s.H + h) * D + lane * PER;
  if constexpr (DENSE) {
    dense_fold<PER>(ds, (size_t)(b * T + i) * s.H + h, M, L, acc, lane, dst);
  } else {
    const float inv = 1.f / L;
#pragma unroll
    for (int e = 0; e < PER; e += 2) {
      *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    }
  }
}

// Dense attention, chunk c: blocks 16c .. 16c+15 of every query, those past
// its local block as -1.
__global__ void dense_sel_kernel(Shape s, Positions pos, int chunk, int32_t* __restrict__ sel) {
  const int64_t n = (int64_t)s.B * s.T * s.G * kTopk;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(e % kTopk);
    const int64_t r = e / kTopk / s.G;       // b * T + i
    const int b = (int)(r / s.T), i = (int)(r % s.T);
    const int64_t lb = ((int64_t)pos.q_start[b] + i) / kBlock;
    const int64_t kb = (int64_t)chunk * kTopk + j;
    sel[e] = kb <= lb ? (int32_t)kb : -1;
  }
}

// topk_merge for at most kSmallLists lists per row: one thread per (pass row,
// group) keeps the head of every list in registers and takes the best head 15
// times.  Same result as topk_merge_kernel; more rows in flight.
constexpr int kSmallLists = 8;
__global__ void __launch_bounds__(256) topk_merge_small_kernel(
    Shape s, Positions pos, int T, int t0, int Tp, int bps, int nsplit, int nrows,
    const Cand* __restrict__ cand, int32_t* __restrict__ sel) {
  const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= (int64_t)nrows * s.G) return;
  const int row = (int)(gi / s.G), g = (int)(gi % s.G);
  const int b = row / Tp, i = t0 + row % Tp;
  const int64_t t = (int64_t)pos.q_start[b] + i;
  const int lb = (int)(t / kBlock);
  const int nvalid = (lb + bps - 1) / bps;
  const Cand* base = cand + (size_t)row * nsplit * s.G * kCand + (size_t)g * kCand;
  const size_t lstride = (size_t)s.G * kCand;
  float hs[kSmallLists];
  int hi[kSmallLists], cur[kSmallLists];
#pragma unroll
  for (int k = 0; k < kSmallLists; ++k) {
    cur[k] = 0;
    hs[k] = -INFINITY;
    hi[k] = INT_MAX;
    if (k < nvalid) {
      const Cand c = base[(size_t)k * lstride];
      hs[k] = c.score;
      hi[k] = c.id;
    }
  }
  int keys[kTopk];
#pragma unroll
  for (int r = 0; r < kCand; ++r) {
    int bk = 0;
    float bs = hs[0];
    int bid = hi[0];
#pragma unroll
    for (int k = 1; k < kSmallLists; ++k)
      if (cand_better(hs[k], hi[k], bs, bid)) {
        bs = hs[k];
        bid = hi[k];
        bk = k;
      }
    int wi = INT_MAX;
#pragma unroll
    for (int k = 0; k < kSmallLists; ++k) {
      if (k == bk) {
        wi = hi[k];
        ++cur[k];
        Cand c = Cand{-INFINITY, INT_MAX};
        if (cur[k] < kCand && wi != INT_MAX) c = base[(size_t)k * lstride + cur[k]];
        hs[k] = c.score;
        hi[k] = c.id;
      }
    }
    keys[r] = r < lb ? wi : INT_MAX;
  }
  keys[kCand] = lb;
  // ascending ids, -1 padding last: each key goes to its rank
  int32_t* out = sel + ((size_t)(b * T + i) * s.G + g) * kTopk;
#pragma unroll
  for (int j = 0; j < kTopk; ++j) {
    int rank = 0;
#pragma unroll
    for (int k = 0; k < kTopk; ++k) rank += (keys[k] < keys[j]) || (keys[k] == keys[j] && k < j);
    out[rank] = keys[j] == INT_MAX ? -1 : keys[j];
  }
}

int pick_bps(int max_lb) {
  int bps = 64;
  while ((max_lb + bps - 1) / bps > kMaxSplits && bps < kMaxBps) bps *= 2;
  return bps;
}

}  // namespace

int max_local_block(const Shape& s, const Positions& pos, int t0, int t1) {
  int m = 0;
  for (int b = 0; b < s.B; ++b) {
    const int64_t t = (int64_t)pos.q_start[b] + t1 - 1;
    const int lb = (int)(t / kBlock);
    if (lb > m) m = lb;
  }
  (void)t0;
  return m;
}

// Capacity bound for any context up to max_lb blocks: a launch uses
// ceil(lb / pick_bps(lb)) <= min(kMaxSplits, ceil(lb / 64)) splits, which is
// monotone in lb.
size_t index_stream_cand_entries(const Shape& s, int rows, int max_lb) {
  int nsplit = (max_lb + 63) / 64;
  if (nsplit > kMaxSplits) nsplit = kMaxSplits;
  return (size_t)rows * (nsplit > 0 ? nsplit : 1) * s.G * kCand;
}

size_t attn_stream_part_rows(const Shape& s, int rows) { return (size_t)rows * s.H * kTopk; }

cudaError_t launch_index_stream(const Shape& s, const Positions& pos, int t0, int t1,
                                const uint16_t* q_idx, const uint16_t* k_idx, int32_t* sel,
                                const Workspace& ws, cudaStream_t st) {
  const int Tp = t1 - t0;
  const int rows = s.B * Tp;
  if (rows <= 0) return cudaSuccess;
  const int max_lb = max_local_block(s, pos, t0, t1);
  const int bps = pick_bps(max_lb);
  const int nsplit = max_lb > 0 ? (max_lb + bps - 1) / bps : 0;
  if (nsplit > 0) {
    note_launches(1);
    dim3 grid(nsplit, rows);
    if (s.Di == 64)
      index_stream_kernel<64><<<grid, kIdxWarps * 32, 0, st>>>(s, pos, s.T, t0, Tp, bps, nsplit,
                                                               q_idx, k_idx, ws.cand, ws.status);
    else
      index_stream_kernel<32><<<grid, kIdxWarps * 32, 0, st>>>(s, pos, s.T, t0, Tp, bps, nsplit,
                                                               q_idx, k_idx, ws.cand, ws.status);
  }
  return launch_topk_merge(s, pos, t0, t1, bps, nsplit > 0 ? nsplit : 1, ws.cand, sel, st);
}

cudaError_t launch_topk_merge(const Shape& s, const Positions& pos, int t0, int t1, int bps,
                              int nsplit, const Cand* cand, int32_t* sel, cudaStream_t st) {
  const int Tp = t1 - t0;
  const int rows = s.B * Tp;
  if (rows <= 0) return cudaSuccess;
  const int64_t warps = (int64_t)rows * s.G;
  const int max_lb = max_local_block(s, pos, t0, t1);
  note_launches(1);
  if ((max_lb + bps - 1) / bps <= kSmallLists)
    topk_merge_small_kernel<<<(unsigned)((warps + 255) / 256), 256, 0, st>>>(
        s, pos, s.T, t0, Tp, bps, nsplit, rows, cand, sel);
  else
    topk_merge_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(s, pos, s.T, t0, Tp, bps,
                                                                 nsplit, rows, cand, sel);
  return cudaGetLastError();
}

cudaError_t launch_dense_sel(const Shape& s, const Positions& pos, int chunk, int32_t* sel,
                             cudaStream_t st) {
  const int64_t n = (int64_t)s.B * s.T * s.G * kTopk;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256;
  note_launches(1);
  dense_sel_kernel<<<(unsigned)(blocks < 65536 ? blocks : 65536), 256, 0, st>>>(s, pos, chunk,
                                                                               sel);
  return cudaGetLastError();
}

namespace {

// Parts per (row, group) of the streaming attention: of 1, 2, 4, 8 and 16,
// the one whose round-robin deal leaves the busiest CTA the least work,
// counting a selected block as 8 and an item's own cost (its query copy, its
// partials written and merged) as 1; ties go to fewer parts.
int attn_stream_parts(int units, int ctas) {
  int best = 1;
  int64_t best_load = INT64_MAX;
  for (int p = 1; p <= kTopk; p *= 2) {
    const int64_t items = (int64_t)units * p;
    const int64_t load = (items + ctas - 1) / ctas * (8 * (kTopk / p) + 1);
    if (load < best_load) {
      best_load = load;
      best = p;
    }
  }
  return best;
}

template <int D, int NTH>
cudaError_t launch_attn_dec(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecArgs& a,
                            int grid, cudaStream_t st) {
  using C = DecCfg<D, NTH>;
  cudaError_t e = cudaFuncSetAttribute(attn_dec_kernel<D, NTH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  attn_dec_kernel<D, NTH><<<grid, kDecThreads, C::kSmem, st>>>(tm_k, tm_v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_stream(const Shape& s, const Positions& pos, int t0, int t1,
                               const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* sel, uint16_t* out, const Workspace& ws,
                               cudaStream_t st, const DenseStep* dense) {
  const int Tp = t1 - t0;
  const int rows = s.B * Tp;
  if (rows <= 0) return cudaSuccess;
  const int hpg = s.H / s.G;
  // K and V as (D dims, G heads, cache tokens); one box = 64 dims x 128
  // tokens of one head, the 128-byte swizzle the consumers index
  CUtensorMap tm_k, tm_v;
  {
    cuuint64_t dims[3] = {(cuuint64_t)s.D, (cuuint64_t)s.G, (cuuint64_t)(s.cache_blocks() * kBlock)};
    cuuint64_t strides[2] = {(cuuint64_t)s.D * 2, (cuuint64_t)s.G * s.D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kBlock};
    if (!encode_bf16_map(&tm_k, k, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_map(&tm_v, v, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const int ctas = sm_count();
  const int units = rows * s.G;
  DecArgs a;
  a.s = s;
  a.pos = pos;
  a.T = s.T;
  a.t0 = t0;
  a.Tp = Tp;
  a.nparts = attn_stream_parts(units, ctas);
  a.spp = kTopk / a.nparts;
  a.nitems = units * a.nparts;
  a.q = q;
  a.sel = sel;
  a.part_o = ws.part_o;
  a.part_ml = ws.part_ml;
  a.status = ws.status;
  a.wait_polls = debug_wait_polls();
  const int grid = a.nitems < ctas ? a.nitems : ctas;
  note_launches(2);
  cudaError_t e;
  if (s.D == 128)
    e = hpg <= 8 ? launch_attn_dec<128, 1>(tm_k, tm_v, a, grid, st)
                 : launch_attn_dec<128, 2>(tm_k, tm_v, a, grid, st);
  else
    e = hpg <= 8 ? launch_attn_dec<64, 1>(tm_k, tm_v, a, grid, st)
                 : launch_attn_dec<64, 2>(tm_k, tm_v, a, grid, st);
  if (e != cudaSuccess) return e;
  const int warps = rows * s.H;
  const DenseStep ds = dense ? *dense : DenseStep{};
#define MSA_ATTN_MERGE(DD)                                                                      \
  if (dense)                                                                                    \
    attn_merge_kernel<DD, true><<<(warps + 7) / 8, 256, 0, st>>>(s, s.T, t0, Tp, rows,          \
                                                                 a.nparts, ws.part_o,           \
                                                                 ws.part_ml, out, ds);          \
  else                                                                                          \
    attn_merge_kernel<DD, false><<<(warps + 7) / 8, 256, 0, st>>>(s, s.T, t0, Tp, rows,         \
                                                                  a.nparts, ws.part_o,          \
                                                                  ws.part_ml, out, ds)
  if (s.D == 128) {
    MSA_ATTN_MERGE(128);
  } else {
    MSA_ATTN_MERGE(64);
  }
#undef MSA_ATTN_MERGE
  return cudaGetLastError();
}

}  // namespace msa
