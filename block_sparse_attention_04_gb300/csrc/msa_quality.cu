// Selection quality and the index branch's training signal.
//
// Selection quality: how much of the attention the selected blocks recall,
// the evaluation "MiniMax 模型迭代与竞品分析" section 2 asks for when it names
// the indexer's recall as MSA's risk (a block the indexer misses cannot be
// read by the main branch).  For every (query, group) of the call:
//
//   A_h(b)         mass of block b (its tokens <= t) under head h's FULL
//                  causal softmax (every token 0..t, no selection)
//   coverage[h]    sum of A_h(b) over the distinct valid ids of sel
//   dense_sel      the ideal selection under the same rule: the local block
//                  plus the top min(16, lb+1)-1 blocks b < lb by the
//                  group-averaged mass P(b) = mean_h A_h(b), ties to the
//                  lower id, ascending, -1 padded
//   best[h]        sum of A_h(b) over dense_sel
//   hits           |sel intersected with dense_sel|  (recall = hits / |dense_sel|)
//
// Two kernels per pass of at most kQualRows (sequence, query) rows:
//   quality_block   grid (block, group, row): S^T = K Q^T for the block's 128
//                   tokens and the group's heads (mma.sync, fp32), causal
//                   mask, per head the block maximum m (log2 units) and
//                   l = sum 2^(s - m); written to scratch
//   quality_reduce  grid (group, row), 256 threads: per head the global
//                   maximum and normaliser over the blocks, the masses, the
//                   coverage sums, the ideal selection (15 rounds of a
//                   block-wide arg-max) and the hits
#include <climits>

#include "msa_device.cuh"

namespace msa {
namespace {

constexpr int kQualRows = 64;       // (sequence, query) rows per pass
constexpr int kReduceThreads = 256;

int qual_pass_len(int B, int T) {
  int tp = kQualRows / B;
  if (tp < 1) tp = 1;
  return tp < T ? tp : (T > 0 ? T : 1);
}

__device__ __forceinline__ bool better(float s1, int i1, float s2, int i2) {
  return s1 > s2 || (s1 == s2 && i1 < i2);
}

// Index-branch training signal (msa_index_kl): per selected block, besides
// the main branch's statistics, the pooled index score and its first
// maximising token.
struct KlIndex {
  const int32_t* sel;      // [B][T][G][16]
  const uint16_t* q_idx;   // [B][T][G][Di]
  const uint16_t* k_idx;   // [B][max_blocks*128][Di]
  float* z;                // [rows][G][16] pooled score
  int32_t* arg;            // [rows][G][16] maximising token (absolute position)
};

// grid (nbl, G, rows) -- or (16 slots, G, rows) with SEL, over the blocks of
// sel only (statistics then restricted to the selected tokens, as in the main
// branch); 128 threads (4 warps, 32 tokens each).  NTH 8-head column tiles
// cover the group's heads.
template <int D, int NTH, bool SEL>
__global__ void __launch_bounds__(128) quality_block_kernel(
    Shape s, Positions pos, int T, int t0, int Tp, int nbl, const uint16_t* __restrict__ q,
    const uint16_t* __restrict__ kc, float2* __restrict__ ml, KlIndex kx) {
  constexpr int NJ = D / 16;
  constexpr int NU = D / 32;
  constexpr int NH = NTH * 8;
  __shared__ float red[4][NH];
  __shared__ float zred[4];
  __shared__ int ared[4];
  const int g = blockIdx.y, row = blockIdx.z;
  const int b = row / Tp, i = t0 + row % Tp;
  const int64_t t = (int64_t)pos.q_start[b] + i;
  const int H = s.H, G = s.G, hpg = H / G;
  int kb = blockIdx.x;
  if constexpr (SEL) {
    kb = kx.sel[(((size_t)b * T + i) * G + g) * kTopk + blockIdx.x];
    if (kb < 0 || kb > (int)(t / kBlock)) {  // not a candidate: nothing to score
      if (threadIdx.x < hpg)
        ml[(((size_t)row * G + g) * kTopk + blockIdx.x) * hpg + threadIdx.x] =
            make_float2(-INFINITY, 0.f);
      return;
    }
  }
  if (kb > (int)(t / kBlock)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;

  // Q^T fragments (dims x heads): dims permuted the same way as the K rows
  uint32_t bq[NTH][NJ][2];
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt) {
    const int hh = nt * 8 + gq;
    const uint16_t* qr =
        q + ((size_t)(b * T + i) * H + (size_t)g * hpg + (hh < hpg ? hh : 0)) * D;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int base = (tq + 4 * (j >> 1)) * 8 + (j & 1) * 4;
      const uint32_t lo = *reinterpret_cast<const uint32_t*>(qr + base);
      const uint32_t hi = *reinterpret_cast<const uint32_t*>(qr + base + 2);
      bq[nt][j][0] = hh < hpg ? lo : 0u;
      bq[nt][j][1] = hh < hpg ? hi : 0u;
    }
  }
  // this warp's 32 tokens of the block, rows gq and gq + 8 of two 16-row groups
  const size_t tok_stride = (size_t)G * D;
  const uint16_t* kblk = kc + (size_t)((int64_t)b * s.max_blocks + kb) * kBlock * tok_stride +
                        (size_t)g * D;
  uint4 L0[2][NU], L1[2][NU];
#pragma unroll
  for (int mg = 0; mg < 2; ++mg) {
    const uint16_t* k0 = kblk + (size_t)(warp * 32 + mg * 16 + gq) * tok_stride;
    const uint16_t* k1 = k0 + 8 * tok_stride;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      L0[mg][u] = ldg_stream(k0 + (tq + 4 * u) * 8);
      L1[mg][u] = ldg_stream(k1 + (tq + 4 * u) * 8);
    }
  }
  const float sl = s.scale * kLog2e;
  float sc[2][NTH][4];
#pragma unroll
  for (int mg = 0; mg < 2; ++mg)
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int u = j >> 1;
        const bool e = j & 1;
        mma_bf16_16816(acc, e ? L0[mg][u].z : L0[mg][u].x, e ? L1[mg][u].z : L1[mg][u].x,
                       e ? L0[mg][u].w : L0[mg][u].y, e ? L1[mg][u].w : L1[mg][u].y,
                       bq[nt][j][0], bq[nt][j][1]);
      }
      const int64_t tok0 = (int64_t)kb * kBlock + warp * 32 + mg * 16 + gq;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t tok = tok0 + (c >= 2 ? 8 : 0);
        sc[mg][nt][c] = tok <= t ? acc[c] * sl : -INFINITY;
      }
    }
  // per head (column): block maximum, then the sum of 2^(s - m)
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
#pragma unroll
  for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = 0.f;
#pragma unroll
      for (int mg = 0; mg < 2; ++mg)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) l += ex2(sc[mg][nt][e + 2 * rr] - mh[nt][e]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (gq == 0) red[warp][nt * 8 + 2 * tq + e] = l;
    }
  __syncthreads();
  if (threadIdx.x < 32 && gq == 0) {
    float2* dst = ml + (((size_t)row * G + g) * (SEL ? kTopk : nbl) + (SEL ? blockIdx.x : kb)) * hpg;
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = nt * 8 + 2 * tq + e;
        if (h < hpg)
          dst[h] = make_float2(mh[nt][e], red[0][h] + red[1][h] + red[2][h] + red[3][h]);
      }
  }
  if constexpr (SEL) {
    // pooled index score of the block: each thread scores one token <= t;
    // the maximum goes to the first token that reaches it
    const int tok = kb * kBlock + threadIdx.x;
    float zt = -INFINITY;
    if (tok <= t) {
      const uint16_t* qi = kx.q_idx + (((size_t)b * T + i) * G + g) * s.Di;
      const uint16_t* kr = kx.k_idx + ((size_t)b * s.max_blocks * kBlock + tok) * s.Di;
      zt = 0.f;
      for (int d = 0; d < s.Di; d += 8) {
        const uint4 a4 = *reinterpret_cast<const uint4*>(qi + d);
        const uint4 k4 = *reinterpret_cast<const uint4*>(kr + d);
        zt = fmaf(bf16lo(a4.x), bf16lo(k4.x), zt);
        zt = fmaf(bf16hi(a4.x), bf16hi(k4.x), zt);
        zt = fmaf(bf16lo(a4.y), bf16lo(k4.y), zt);
        zt = fmaf(bf16hi(a4.y), bf16hi(k4.y), zt);
        zt = fmaf(bf16lo(a4.z), bf16lo(k4.z), zt);
        zt = fmaf(bf16hi(a4.z), bf16hi(k4.z), zt);
        zt = fmaf(bf16lo(a4.w), bf16lo(k4.w), zt);
        zt = fmaf(bf16hi(a4.w), bf16hi(k4.w), zt);
      }
    }
    int at = tok;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float z2 = __shfl_xor_sync(0xffffffffu, zt, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, at, o);
      if (z2 > zt || (z2 == zt && a2 < at)) {
        zt = z2;
        at = a2;
      }
    }
    if (lane == 0) {
      zred[warp] = zt;
      ared[warp] = at;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < 4; ++w)
        if (zred[w] > zt) {  // warps hold increasing tokens: ties keep the earlier
          zt = zred[w];
          at = ared[w];
        }
      const size_t o = ((size_t)row * G + g) * kTopk + blockIdx.x;
      kx.z[o] = zt;
      kx.arg[o] = at;
    }
  }
}

// Block-wide arg-best of (score, id) pairs held one per thread.
__device__ __forceinline__ void block_argbest(float& sc, int& id, float* ws, int* wi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, sc, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, id, o);
    if (better(s2, i2, sc, id)) {
      sc = s2;
      id = i2;
    }
  }
  if (lane == 0) {
    ws[warp] = sc;
    wi[warp] = id;
  }
  __syncthreads();
  sc = ws[0];
  id = wi[0];
#pragma unroll
  for (int w = 1; w < kReduceThreads / 32; ++w)
    if (better(ws[w], wi[w], sc, id)) {
      sc = ws[w];
      id = wi[w];
    }
  __syncthreads();
}

// Block-wide reduction (max or sum) of up to 16 per-head values.
template <bool MAX>
__device__ __forceinline__ void block_reduce16(float (&v)[16], float (*sh)[16]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    float x = v[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x, o);
      x = MAX ? fmaxf(x, y) : x + y;
    }
    if (lane == 0) sh[warp][h] = x;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    float x = sh[0][h];
#pragma unroll
    for (int w = 1; w < kReduceThreads / 32; ++w) x = MAX ? fmaxf(x, sh[w][h]) : x + sh[w][h];
    v[h] = x;
  }
  __syncthreads();
}

// grid (G, rows); kReduceThreads threads.
__global__ void __launch_bounds__(kReduceThreads) quality_reduce_kernel(
    Shape s, Positions pos, int T, int t0, int Tp, int nbl, const int32_t* __restrict__ sel,
    const float2* __restrict__ ml, float* __restrict__ pmass, float* __restrict__ coverage,
    float* __restrict__ best, int32_t* __restrict__ dense_sel, int32_t* __restrict__ hits) {
  __shared__ float sh[kReduceThreads / 32][16];
  __shared__ float wsc[kReduceThreads / 32];
  __shared__ int wid[kReduceThreads / 32];
  __shared__ int chosen[kTopk];
  const int g = blockIdx.x, row = blockIdx.y;
  const int b = row / Tp, i = t0 + row % Tp;
  const int64_t t = (int64_t)pos.q_start[b] + i;
  const int lb = (int)(t / kBlock), nblk = lb + 1;
  const int H = s.H, G = s.G, hpg = H / G;
  const float2* m = ml + ((size_t)row * G + g) * nbl * hpg;
  float* P = pmass + ((size_t)row * G + g) * nbl;
  const size_t orow = (size_t)b * T + i;

  // per head: the maximum over blocks, then the normaliser
  float M[16], Z[16];
#pragma unroll
  for (int h = 0; h < 16; ++h) M[h] = -INFINITY;
  for (int k = threadIdx.x; k < nblk; k += kReduceThreads)
#pragma unroll
    for (int h = 0; h < 16; ++h)
      if (h < hpg) M[h] = fmaxf(M[h], m[(size_t)k * hpg + h].x);
  block_reduce16<true>(M, sh);
#pragma unroll
  for (int h = 0; h < 16; ++h) Z[h] = 0.f;
  for (int k = threadIdx.x; k < nblk; k += kReduceThreads)
#pragma unroll
    for (int h = 0; h < 16; ++h)
      if (h < hpg) {
        const float2 x = m[(size_t)k * hpg + h];
        Z[h] += ex2(x.x - M[h]) * x.y;
      }
  block_reduce16<false>(Z, sh);
  // group-averaged mass of every block
  const float inv_hpg = 1.f / (float)hpg;
  for (int k = threadIdx.x; k < nblk; k += kReduceThreads) {
    float p = 0.f;
#pragma unroll
    for (int h = 0; h < 16; ++h)
      if (h < hpg) {
        const float2 x = m[(size_t)k * hpg + h];
        p += ex2(x.x - M[h]) * x.y / Z[h];
      }
    P[k] = p * inv_hpg;
  }
  __syncthreads();
  // the ideal selection: local block, then the best blocks b < lb by mass
  const int nsel = nblk < kTopk ? nblk : kTopk;
  float last_s = INFINITY;
  int last_i = -1;
  for (int r = 0; r < nsel - 1; ++r) {
    float bs = -INFINITY;
    int bi = INT_MAX;
    for (int k = threadIdx.x; k < lb; k += kReduceThreads) {
      const float p = P[k];
      const bool eligible = p < last_s || (p == last_s && k > last_i);
      if (eligible && better(p, k, bs, bi)) {
        bs = p;
        bi = k;
      }
    }
    block_argbest(bs, bi, wsc, wid);
    if (threadIdx.x == 0) chosen[r] = bi;
    last_s = bs;
    last_i = bi;
  }
  if (threadIdx.x == 0) chosen[nsel - 1] = lb;
  __syncthreads();
  // outputs: one thread per head for the mass sums, thread 0 for the ids
  const int32_t* sg = sel + (orow * G + g) * kTopk;
  if ((int)threadIdx.x < hpg) {
    const int h = threadIdx.x;
    float c = 0.f, cb = 0.f;
    for (int j = 0; j < kTopk; ++j) {
      const int id = sg[j];
      bool fresh = id >= 0 && id <= lb;
      for (int u = 0; u < j && fresh; ++u) fresh = sg[u] != id;
      if (fresh) {
        const float2 x = m[(size_t)id * hpg + h];
        c += ex2(x.x - M[h]) * x.y / Z[h];
      }
    }
    for (int j = 0; j < nsel; ++j) {
      const float2 x = m[(size_t)chosen[j] * hpg + h];
      cb += ex2(x.x - M[h]) * x.y / Z[h];
    }
    coverage[orow * H + (size_t)g * hpg + h] = c;
    best[orow * H + (size_t)g * hpg + h] = cb;
  }
  if (threadIdx.x == 32) {
    int ids[kTopk];
#pragma unroll
    for (int j = 0; j < kTopk; ++j) ids[j] = j < nsel ? chosen[j] : INT_MAX;
    // ascending (16 entries, insertion sort)
    for (int j = 1; j < kTopk; ++j) {
      const int x = ids[j];
      int u = j - 1;
      while (u >= 0 && ids[u] > x) {
        ids[u + 1] = ids[u];
        --u;
      }
      ids[u + 1] = x;
    }
    int32_t* ds = dense_sel + (orow * G + g) * kTopk;
    int nh = 0;
    for (int j = 0; j < kTopk; ++j) {
      ds[j] = ids[j] == INT_MAX ? -1 : ids[j];
      const int id = sg[j];
      bool fresh = id >= 0 && id <= lb;
      for (int u = 0; u < j && fresh; ++u) fresh = sg[u] != id;
      if (fresh)
        for (int k = 0; k < nsel; ++k) nh += chosen[k] == id;
    }
    hits[orow * G + g] = nh;
  }
}

// grid (rows in the pass), G warps per CTA: one warp per (query, group), lane
// j holding candidate slot j.  P from the slots' (m, l) statistics, Q from
// their pooled scores, the loss, dQ_idx (written) and dK_idx (accumulated at
// each block's maximising token with atomic adds).
__global__ void __launch_bounds__(256) kl_reduce_kernel(Shape s, Positions pos, int T, int t0,
                                                        int Tp, const float2* __restrict__ ml,
                                                        KlIndex kx, float* __restrict__ kl,
                                                        float* __restrict__ dq_idx,
                                                        float* __restrict__ dk_idx) {
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (g >= s.G) return;
  const int row = blockIdx.x;
  const int b = row / Tp, i = t0 + row % Tp;
  const int64_t t = (int64_t)pos.q_start[b] + i;
  const int lb = (int)(t / kBlock);
  const int hpg = s.H / s.G, Di = s.Di;
  const size_t orow = ((size_t)b * T + i) * s.G + g;
  // candidates: the distinct ids of sel in [0, lb], in slot order
  const int id = lane < kTopk ? kx.sel[orow * kTopk + lane] : -1;
  bool valid = id >= 0 && id <= lb;
  for (int u = 0; u < kTopk; ++u) {
    const int idu = __shfl_sync(0xffffffffu, id, u);
    if (u < lane && idu == id) valid = false;
  }
  const size_t srow = ((size_t)row * s.G + g) * kTopk + lane;
  // teacher: the main branch's softmax mass per candidate, averaged over heads
  float P = 0.f;
  for (int h = 0; h < hpg; ++h) {
    float2 x = make_float2(-INFINITY, 0.f);
    if (valid) x = ml[srow * hpg + h];
    float M = x.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = valid ? ex2(x.x - M) * x.y : 0.f;
    float Z = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    P += w / Z;
  }
  P /= (float)hpg;
  // student: softmax of the pooled index scores over the same candidates
  const float z = valid ? kx.z[srow] : -INFINITY;
  float zm = z;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, o));
  const float e = valid ? expf(z - zm) : 0.f;
  float se = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
  const float Q = e / se;
  float term = (valid && P > 0.f) ? P * (logf(P) - logf(Q)) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
  if (lane == 0) kl[orow] = term;
  // gradients: dz_j = Q_j - P_j through each block's maximising token
  const float dz = valid ? Q - P : 0.f;
  const int at = valid ? kx.arg[srow] : 0;
  const uint16_t* qi = kx.q_idx + orow * Di;
  const uint16_t* kseq = kx.k_idx + (size_t)b * s.max_blocks * kBlock * Di;
  float* dkseq = dk_idx + (size_t)b * s.max_blocks * kBlock * Di;
  for (int d = lane; d < Di; d += 32) {
    const float qd = bf16lo((uint32_t)qi[d]);
    float acc = 0.f;
    for (int j = 0; j < kTopk; ++j) {
      const float dzj = __shfl_sync(0xffffffffu, dz, j);
      const int aj = __shfl_sync(0xffffffffu, at, j);
      if (dzj != 0.f) {
        acc = fmaf(dzj, bf16lo((uint32_t)kseq[(size_t)aj * Di + d]), acc);
        atomicAdd(dkseq + (size_t)aj * Di + d, dzj * qd);
      }
    }
    dq_idx[orow * Di + d] = acc;
  }
}

struct QualLayout {
  size_t ml_off, p_off, total;
};

QualLayout qual_layout(const Shape& s) {
  const size_t rows = (size_t)s.B * qual_pass_len(s.B, s.T);
  const size_t hpg = (size_t)(s.H / s.G);
  QualLayout L{};
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  L.ml_off = 0;
  L.p_off = al(rows * s.G * s.max_blocks * hpg * sizeof(float2));
  L.total = L.p_off + al(rows * s.G * s.max_blocks * sizeof(float));
  return L;
}

constexpr int kKlRows = 8192;   // (sequence, query) rows per pass of msa_index_kl

int kl_pass_len(int B, int T) {
  int tp = kKlRows / B;
  if (tp < 1) tp = 1;
  return tp < T ? tp : (T > 0 ? T : 1);
}

struct KlLayout {
  size_t ml_off, z_off, a_off, total;
};

KlLayout kl_layout(const Shape& s) {
  const size_t rows = (size_t)s.B * kl_pass_len(s.B, s.T);
  const size_t slots = rows * s.G * kTopk;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  KlLayout L{};
  L.ml_off = 0;
  L.z_off = al(slots * (s.H / s.G) * sizeof(float2));
  L.a_off = L.z_off + al(slots * sizeof(float));
  L.total = L.a_off + al(slots * sizeof(int32_t));
  return L;
}

}  // namespace

size_t quality_workspace_bytes(const Shape& s) { return qual_layout(s).total; }

size_t kl_workspace_bytes(const Shape& s) { return kl_layout(s).total; }

cudaError_t launch_index_kl(const Shape& s, const Positions& pos, const uint16_t* q_idx,
                            const uint16_t* k_idx, const uint16_t* q, const uint16_t* k,
                            const int32_t* sel, float* kl, float* dq_idx, float* dk_idx, char* ws,
                            cudaStream_t st) {
  const KlLayout lay = kl_layout(s);
  float2* ml = reinterpret_cast<float2*>(ws + lay.ml_off);
  KlIndex kx{sel, q_idx, k_idx, reinterpret_cast<float*>(ws + lay.z_off),
             reinterpret_cast<int32_t*>(ws + lay.a_off)};
  const int hpg = s.H / s.G;
  const int tp_max = kl_pass_len(s.B, s.T);
  for (int t0 = 0; t0 < s.T; t0 += tp_max) {
    const int Tp = tp_max < s.T - t0 ? tp_max : s.T - t0;
    const int rows = s.B * Tp;
    dim3 g1(kTopk, s.G, rows);
    note_launches(2);
#define MSA_KL_BLOCK(DD, NT)                                                                 \
  quality_block_kernel<DD, NT, true><<<g1, 128, 0, st>>>(s, pos, s.T, t0, Tp, kTopk, q, k, ml, kx)
    if (s.D == 128) {
      if (hpg <= 8) MSA_KL_BLOCK(128, 1); else MSA_KL_BLOCK(128, 2);
    } else {
      if (hpg <= 8) MSA_KL_BLOCK(64, 1); else MSA_KL_BLOCK(64, 2);
    }
#undef MSA_KL_BLOCK
    kl_reduce_kernel<<<rows, 32 * s.G, 0, st>>>(s, pos, s.T, t0, Tp, ml, kx, kl, dq_idx, dk_idx);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_quality(const Shape& s, const Positions& pos, const uint16_t* q,
                           const uint16_t* k, const int32_t* sel, float* coverage, float* best,
                           int32_t* dense_sel, int32_t* hits, char* ws, cudaStream_t st) {
  const QualLayout lay = qual_layout(s);
  float2* ml = reinterpret_cast<float2*>(ws + lay.ml_off);
  float* pm = reinterpret_cast<float*>(ws + lay.p_off);
  const int hpg = s.H / s.G;
  const int tp_max = qual_pass_len(s.B, s.T);
  for (int t0 = 0; t0 < s.T; t0 += tp_max) {
    const int Tp = tp_max < s.T - t0 ? tp_max : s.T - t0;
    const int rows = s.B * Tp;
    const int nbl = max_local_block(s, pos, t0, t0 + Tp) + 1;
    dim3 g1(nbl, s.G, rows);
    note_launches(2);
#define MSA_QUAL_BLOCK(DD, NT)                                                              \
  quality_block_kernel<DD, NT, false><<<g1, 128, 0, st>>>(s, pos, s.T, t0, Tp, nbl, q, k, ml,   \
                                                          KlIndex{})
    if (s.D == 128) {
      if (hpg <= 8) MSA_QUAL_BLOCK(128, 1); else MSA_QUAL_BLOCK(128, 2);
    } else {
      if (hpg <= 8) MSA_QUAL_BLOCK(64, 1); else MSA_QUAL_BLOCK(64, 2);
    }
#undef MSA_QUAL_BLOCK
    quality_reduce_kernel<<<dim3(s.G, rows), kReduceThreads, 0, st>>>(
        s, pos, s.T, t0, Tp, nbl, sel, ml, pm, coverage, best, dense_sel, hits);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace msa
