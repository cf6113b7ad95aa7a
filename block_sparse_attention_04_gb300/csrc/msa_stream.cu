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
//   attn_stream   step 4 for one selected block of one (query, group): scores
//                 of all heads of the group (mma), block-local softmax
//                 statistics, P.V (mma), written as an unnormalised partial.
//   attn_merge    combines the <= 16 block partials of each (query, head)
//                 (log-sum-exp merge) into the bf16 output.
#include <cfloat>
#include <climits>

#include "msa_device.cuh"

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
  // (a block-table entry outside the pool is flagged and block 0 read instead)
#define MSA_IDX_LOAD(IT, X0, X1)                                                        \
  do {                                                                                  \
    const int blk_ = blk0 + warp + ((IT) / SPB) * kIdxWarps;                            \
    const int64_t pb_ = cache_block(s, b, blk_, status);                                \
    const uint16_t* r_ =                                                                \
        k_idx + ((size_t)(pb_ < 0 ? 0 : pb_) * kBlock + ((IT) % SPB) * 16 + gq) * DI;    \
    _Pragma("unroll") for (int u_ = 0; u_ < NU; ++u_) {                                 \
      X0[u_] = ldg_stream(r_ + (tq + 4 * u_) * 8);                                      \
      X1[u_] = ldg_stream(r_ + 8 * DI + (tq + 4 * u_) * 8);                             \
    }                                                                                   \
  } while (0)
  if (n > 0) MSA_IDX_LOAD(0, C0, C1);
  float m0 = -INFINITY, m1 = -INFINITY;
  for (int it = 0; it < n; ++it) {
    uint4 N0[NU], N1[NU];
    if (it + 1 < n) {
      MSA_IDX_LOAD(it + 1, N0, N1);
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
// attn_stream: grid (16 slots, G, pass rows); 128 threads (4 warps).
// NTH = 8-head column tiles per group (heads per group <= 8 * NTH).
template <int D, int NTH>
__global__ void __launch_bounds__(128) attn_stream_kernel(
    Shape s, Positions pos, int T, int t0, int Tp, const uint16_t* __restrict__ q,
    const uint16_t* __restrict__ kc, const uint16_t* __restrict__ vc,
    const int32_t* __restrict__ sel, float* __restrict__ part_o, float* __restrict__ part_ml,
    int* __restrict__ status) {
  constexpr int NJ = D / 16;          // k-steps of the score mma
  constexpr int NU = D / 32;          // 16-byte loads per K row and thread
  constexpr int VSTR = D + 8;         // padded V row (elements)
  constexpr int PSTR = kBlock + 8;    // padded P row (elements)
  constexpr int NH = NTH * 8;
  __shared__ __align__(16) uint16_t vs[kBlock * VSTR];
  __shared__ __align__(16) uint16_t ps[NH * PSTR];
  __shared__ float red[4][NH];

  const int slot = blockIdx.x, g = blockIdx.y, row = blockIdx.z;
  const int b = row / Tp, i = t0 + row % Tp;
  const int64_t t = (int64_t)pos.q_start[b] + i;
  const int lb = (int)(t / kBlock);
  const int H = s.H, G = s.G, hpg = H / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const size_t ml_base = ((size_t)row * H + (size_t)g * hpg) * kTopk + slot;

  // Q^T fragments (dims x heads), same dim permutation as the K fragments;
  // loaded before the selection so that the two loads overlap
  uint32_t bq[NTH][NJ][2];
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt) {
    const int hh = nt * 8 + gq;
    const uint16_t* qr = q + ((size_t)(b * T + i) * H + (size_t)g * hpg + (hh < hpg ? hh : 0)) * D;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int base = (tq + 4 * (j >> 1)) * 8 + (j & 1) * 4;
      uint32_t lo = *reinterpret_cast<const uint32_t*>(qr + base);
      uint32_t hi = *reinterpret_cast<const uint32_t*>(qr + base + 2);
      bq[nt][j][0] = hh < hpg ? lo : 0u;
      bq[nt][j][1] = hh < hpg ? hi : 0u;
    }
  }

  int kb = sel[((size_t)(b * T + i) * G + g) * kTopk + slot];
  if (kb > lb || kb >= s.max_blocks) {
    if (threadIdx.x == 0) flag_invalid(status);
    kb = -1;
  }
  int64_t pb = -1;   // the cache block holding it
  if (kb >= 0) {
    pb = cache_block(s, b, kb, nullptr);
    if (pb < 0) {
      if (threadIdx.x == 0) flag_invalid(status);
      kb = -1;
    }
  }
  if (kb < 0) {
    for (int h = threadIdx.x; h < hpg; h += blockDim.x) {
      part_ml[(ml_base + (size_t)h * kTopk) * 2 + 0] = -INFINITY;
      part_ml[(ml_base + (size_t)h * kTopk) * 2 + 1] = 0.f;
    }
    return;
  }

  const size_t tok_stride = (size_t)G * D;
  const uint16_t* kblk = kc + (size_t)pb * kBlock * tok_stride + (size_t)g * D;
  const uint16_t* vblk = vc + (size_t)pb * kBlock * tok_stride + (size_t)g * D;

  // scores S^T[token][head] for this warp's 32 tokens
  float sc[2][NTH][4];
  const float qk_scale = s.scale * kLog2e;
  // the warp's whole 32-token K slice is requested before the first score MMA
  // and before the V copy, which is needed later: twice the bytes in flight of
  // loading K in 16-token halves, and K first in the memory queue (measured
  // 0.128 -> 0.101 ms on the 64 x 256K decode batch, although the registers
  // this holds leave 4 CTAs per SM instead of 6)
  uint4 LL0[2][NU], LL1[2][NU];
#pragma unroll
  for (int mg = 0; mg < 2; ++mg) {
    const uint16_t* k0 = kblk + (size_t)(warp * 32 + mg * 16 + gq) * tok_stride;
    const uint16_t* k1 = k0 + 8 * tok_stride;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      LL0[mg][u] = ldg_stream(k0 + (tq + 4 * u) * 8);
      LL1[mg][u] = ldg_stream(k1 + (tq + 4 * u) * 8);
    }
  }
  // V block -> shared memory (lands during the score computation)
  for (int c = threadIdx.x; c < kBlock * (D / 8); c += blockDim.x) {
    const int r = c / (D / 8), ch = c % (D / 8);
    cp_async_16(smem_u32(vs + r * VSTR + ch * 8), vblk + r * tok_stride + ch * 8);
  }
  cp_async_commit();

#pragma unroll
  for (int mg = 0; mg < 2; ++mg) {
    const int r0 = warp * 32 + mg * 16 + gq;
    const uint4* L0 = LL0[mg];
    const uint4* L1 = LL1[mg];
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int u = j >> 1;
        const bool e = j & 1;
        mma_bf16_16816(acc, e ? L0[u].z : L0[u].x, e ? L1[u].z : L1[u].x,
                       e ? L0[u].w : L0[u].y, e ? L1[u].w : L1[u].y, bq[nt][j][0],
                       bq[nt][j][1]);
      }
      const int64_t tok0 = (int64_t)kb * kBlock + r0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t tok = tok0 + (c >= 2 ? 8 : 0);
        sc[mg][nt][c] = tok <= t ? acc[c] * qk_scale : -INFINITY;
      }
    }
  }

  // block-local max per head
  float mh[NTH][2];
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float m = fmaxf(fmaxf(sc[0][nt][e], sc[0][nt][e + 2]), fmaxf(sc[1][nt][e], sc[1][nt][e + 2]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (gq == 0) red[warp][nt * 8 + 2 * tq + e] = m;
    }
  __syncthreads();
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = nt * 8 + 2 * tq + e;
      mh[nt][e] = fmaxf(fmaxf(red[0][h], red[1][h]), fmaxf(red[2][h], red[3][h]));
    }
  __syncthreads();

  // p = 2^(s - m) -> bf16 P[head][token]; row sums
  float lh[NTH][2];
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
          const float p = ex2(sc[mg][nt][e + 2 * rr] - mh[nt][e]);
          sum += p;
          ps[h * PSTR + warp * 32 + mg * 16 + gq + 8 * rr] = (uint16_t)f32_to_bf16_rne(p);
        }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      lh[nt][e] = sum;
      if (gq == 0) red[warp][h] = sum;
    }
  cp_async_wait<0>();
  __syncthreads();

  // O^T[dim][head] = V^T P^T; warp w owns dims [w*D/4, (w+1)*D/4)
  constexpr int MGV = D / 64;  // 16-dim groups per warp
  float o[MGV][NTH][4];
#pragma unroll
  for (int mg = 0; mg < MGV; ++mg)
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[mg][nt][c] = 0.f;
  const uint32_t* p32 = reinterpret_cast<const uint32_t*>(ps);
#pragma unroll
  for (int ks = 0; ks < kBlock / 16; ++ks) {
#pragma unroll
    for (int mg = 0; mg < MGV; ++mg) {
      const int dim0 = warp * (D / 4) + mg * 16;
      const int mi = lane >> 3;
      const int tok = ks * 16 + (lane & 7) + ((mi & 2) ? 8 : 0);
      const int dim = dim0 + ((mi & 1) ? 8 : 0);
      uint32_t a[4];
      ldmatrix_x4_trans(a, smem_u32(vs + tok * VSTR + dim));
#pragma unroll
      for (int nt = 0; nt < NTH; ++nt) {
        const int h = nt * 8 + gq;
        const uint32_t b0 = p32[(h * PSTR) / 2 + ks * 8 + tq];
        const uint32_t b1 = p32[(h * PSTR) / 2 + ks * 8 + 4 + tq];
        mma_bf16_16816(o[mg][nt], a[0], a[1], a[2], a[3], b0, b1);
      }
    }
  }

  // partial outputs (unnormalised, relative to the block max)
#pragma unroll
  for (int mg = 0; mg < MGV; ++mg)
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int h = nt * 8 + 2 * tq + (c & 1);
        const int dim = warp * (D / 4) + mg * 16 + gq + (c >= 2 ? 8 : 0);
        if (h < hpg) part_o[(ml_base + (size_t)h * kTopk) * D + dim] = o[mg][nt][c];
      }
  if (threadIdx.x < 32) {
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = nt * 8 + 2 * tq + e;
        const float l = red[0][h] + red[1][h] + red[2][h] + red[3][h];
        if (gq == 0 && h < hpg) {
          part_ml[(ml_base + (size_t)h * kTopk) * 2 + 0] = mh[nt][e];
          part_ml[(ml_base + (size_t)h * kTopk) * 2 + 1] = l;
        }
      }
  }
  (void)lh;
}

// ---------------------------------------------------------------------------
// attn_merge: one warp per (pass row, head).
// DENSE: fold into the dense accumulators instead (one chunk of msa_dense_attn).
template <int D, bool DENSE>
__global__ void __launch_bounds__(256) attn_merge_kernel(
    Shape s, int T, int t0, int Tp, int nrows, const float* __restrict__ part_o,
    const float* __restrict__ part_ml, uint16_t* __restrict__ out, DenseStep ds) {
  constexpr int PER = D / 32;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= nrows * s.H) return;
  const int row = gw / s.H, h = gw % s.H;
  const int b = row / Tp, i = t0 + row % Tp;
  const size_t base = ((size_t)row * s.H + h) * kTopk;
  float m = -INFINITY, l = 0.f;
  if (lane < kTopk) {
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
  for (int j = 0; j < kTopk; ++j) {
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

cudaError_t launch_attn_stream(const Shape& s, const Positions& pos, int t0, int t1,
                               const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* sel, uint16_t* out, const Workspace& ws,
                               cudaStream_t st, const DenseStep* dense) {
  const int Tp = t1 - t0;
  const int rows = s.B * Tp;
  if (rows <= 0) return cudaSuccess;
  const int hpg = s.H / s.G;
  dim3 grid(kTopk, s.G, rows);
  note_launches(2);
#define MSA_ATTN_STREAM(DD, NT)                                                              \
  attn_stream_kernel<DD, NT><<<grid, 128, 0, st>>>(s, pos, s.T, t0, Tp, q, k, v, sel,       \
                                                   ws.part_o, ws.part_ml, ws.status)
  if (s.D == 128) {
    if (hpg <= 8) MSA_ATTN_STREAM(128, 1); else MSA_ATTN_STREAM(128, 2);
  } else {
    if (hpg <= 8) MSA_ATTN_STREAM(64, 1); else MSA_ATTN_STREAM(64, 2);
  }
#undef MSA_ATTN_STREAM
  const int warps = rows * s.H;
  const DenseStep ds = dense ? *dense : DenseStep{};
#define MSA_ATTN_MERGE(DD)                                                                       \
  if (dense)                                                                                     \
    attn_merge_kernel<DD, true><<<(warps + 7) / 8, 256, 0, st>>>(s, s.T, t0, Tp, rows, ws.part_o, \
                                                                 ws.part_ml, out, ds);           \
  else                                                                                           \
    attn_merge_kernel<DD, false><<<(warps + 7) / 8, 256, 0, st>>>(s, s.T, t0, Tp, rows,          \
                                                                  ws.part_o, ws.part_ml, out, ds)
  if (s.D == 128) {
    MSA_ATTN_MERGE(128);
  } else {
    MSA_ATTN_MERGE(64);
  }
#undef MSA_ATTN_MERGE
  return cudaGetLastError();
}

}  // namespace msa
