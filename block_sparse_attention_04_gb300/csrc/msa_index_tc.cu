// Tensor-core index scan for prefill: steps 1-3 of "MiniMax 模型迭代与竞品分析"
// section 2 (global index scoring over the causal context, 128-token block
// max-pooling, top-16 with the local block forced in) for many queries at once.
//
// Rows are (query, group) pairs, r = (b*T + i)*G + g, so one Q_idx tile of
// 128 rows is 128/G queries x G groups and every group reuses the same K_idx
// tile.  One work item = 2 row tiles (256 rows) x one split of at most
// kSplitBlocks key blocks.  Per item and key block (128 keys):
//   warp 0      TMA: the two Q_idx tiles once per item, K_idx tiles through a
//               kStages-deep shared-memory ring;
//   warp 1      tcgen05.mma (M 128, N 128, K Di, bf16 in, fp32 accumulate)
//               for both row tiles into one of two TMEM accumulator stages;
//   warps 2-9   epilogue: tcgen05.ld of the 128 fp32 scores of its row,
//               block maximum (3-input max), insertion into the row's
//               register-resident top-15 (score desc, block id asc).
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
constexpr int kItemRows = 2 * kTileRows;
constexpr int kSplitBlocks = 256;
constexpr int kStages = 6;
constexpr int kThreads = 320;  // 10 warps
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;

template <int DI>
struct IdxCfg {
  static constexpr int kRowBytes = DI * 2;
  static constexpr int kTileBytes = kTileRows * kRowBytes;
  static constexpr uint32_t kSwz = DI == 64 ? kSwizzle128B : kSwizzle64B;
  static constexpr uint32_t kSbo = 8 * kRowBytes;  // one 8-row swizzle atom
  static constexpr int kKSteps = DI / 16;
  static constexpr int kSmemA = 2 * 2 * kTileBytes;         // 2 buffers x 2 row tiles
  static constexpr int kSmemB = kStages * kTileBytes;
  static constexpr int kSmemBar = 256;
  static constexpr int kSmem = kSmemA + kSmemB + kSmemBar + 1024;  // + alignment slack
};

struct IndexTcArgs {
  Shape s;
  Positions pos;
  int npairs;   // item row pairs per sequence
  int nsplit;   // splits per pair (the merge's list count per row)
  int nitems;
  int64_t cap;  // K_idx rows per sequence
  Cand* cand;
  int* status;
};

// Work item -> sequence b, row pair p, split sp and key-block range [k0, k1).
// Pairs are visited last-first (the longest key ranges first).
__device__ __forceinline__ bool item_range(const IndexTcArgs& a, int item, int& b, int& p, int& sp,
                                           int& k0, int& k1) {
  const int per_b = a.npairs * a.nsplit;
  b = item / per_b;
  const int rem = item - b * per_b;
  p = a.npairs - 1 - rem / a.nsplit;
  sp = rem % a.nsplit;
  const int i_last = min(a.s.T - 1, ((p + 1) * kItemRows - 1) / a.s.G);
  const int kb_end = (int)(((int64_t)a.pos.q_start[b] + i_last) / kBlock);
  k0 = sp * kSplitBlocks;
  k1 = min(k0 + kSplitBlocks, kb_end);
  return k0 < k1;
}

template <int DI>
__global__ void __launch_bounds__(kThreads, 1)
    index_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const IndexTcArgs a) {
  using C = IdxCfg<DI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;                 // [abuf][tile][128 rows][DI]
  uint8_t* sB = smem + C::kSmemA;     // [stage][128 keys][DI]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kSmemA + C::kSmemB);
  uint64_t* full = bars;                      // kStages
  uint64_t* empty = bars + kStages;           // kStages
  uint64_t* a_full = bars + 2 * kStages;      // 2
  uint64_t* a_empty = a_full + 2;             // 2
  uint64_t* tm_full = a_empty + 2;            // 2
  uint64_t* tm_empty = tm_full + 2;           // 2
  uint64_t* mma_done = tm_empty + 2;          // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
      mbar_init(&tm_full[i], 1);
      mbar_init(&tm_empty[i], kEpiWarps);
    }
    mbar_init(mma_done, 1);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      int stage = 0, abuf = 0;
      uint32_t sphase = 0, aphase = 0;
      int issued = 0;
      for (int item = blockIdx.x; item < a.nitems && !*abort_flag; item += gridDim.x) {
        int b, p, sp, k0, k1;
        if (!item_range(a, item, b, p, sp, k0, k1)) continue;
        if (!mbar_wait(&a_empty[abuf], aphase ^ 1, a.status)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&a_full[abuf], 2 * C::kTileBytes);
        const int row0 = (b * T) * G + p * kItemRows;
        tma_load_2d(smem_u32(sA + (abuf * 2 + 0) * C::kTileBytes), &tm_q, &a_full[abuf], 0, row0);
        tma_load_2d(smem_u32(sA + (abuf * 2 + 1) * C::kTileBytes), &tm_q, &a_full[abuf], 0,
                    row0 + kTileRows);
        if (++abuf == 2) { abuf = 0; aphase ^= 1; }
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&empty[stage], sphase ^ 1, a.status)) { *abort_flag = 1; break; }
          mbar_arrive_expect_tx(&full[stage], C::kTileBytes);
          tma_load_2d(smem_u32(sB + stage * C::kTileBytes), &tm_k, &full[stage], 0,
                      (int)(b * a.cap + (int64_t)kb * kBlock));
          ++issued;
          if (++stage == kStages) { stage = 0; sphase ^= 1; }
        }
      }
      if (*abort_flag) {
        // drain: wait (bounded) for the loads this thread issued most recently
        int n = issued < kStages ? issued : kStages;
        int st = stage;
        uint32_t ph = sphase;
        for (int k = 0; k < n; ++k) {
          if (st == 0) { st = kStages - 1; ph ^= 1; } else { --st; }
          mbar_wait(&full[st], ph, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
      int stage = 0, abuf = 0, ts = 0;
      uint32_t sphase = 0, aphase = 0, tphase = 0;
      for (int item = blockIdx.x; item < a.nitems && !*abort_flag; item += gridDim.x) {
        int b, p, sp, k0, k1;
        if (!item_range(a, item, b, p, sp, k0, k1)) continue;
        if (!mbar_wait(&a_full[abuf], aphase, a.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + (abuf * 2 + 0) * C::kTileBytes);
        const uint32_t a1 = smem_u32(sA + (abuf * 2 + 1) * C::kTileBytes);
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&full[stage], sphase, a.status) ||
              !mbar_wait(&tm_empty[ts], tphase ^ 1, a.status)) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t bsm = smem_u32(sB + stage * C::kTileBytes);
          const uint32_t d0 = tmem + ts * 256;
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const uint64_t bd = smem_desc(bsm + k * 32, 16, C::kSbo, C::kSwz);
            tc_mma_f16(d0, smem_desc(a0 + k * 32, 16, C::kSbo, C::kSwz), bd, idesc, k > 0);
            tc_mma_f16(d0 + 128, smem_desc(a1 + k * 32, 16, C::kSbo, C::kSwz), bd, idesc, k > 0);
          }
          tc_commit(&empty[stage]);
          tc_commit(&tm_full[ts]);
          if (++stage == kStages) { stage = 0; sphase ^= 1; }
          if (++ts == 2) { ts = 0; tphase ^= 1; }
        }
        if (*abort_flag) break;
        tc_commit(&a_empty[abuf]);
        if (++abuf == 2) { abuf = 0; aphase ^= 1; }
      }
      // all MMAs issued by this thread complete before TMEM is released
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int tile = ew >> 2;
    const int quad = warp & 3;  // TMEM lanes this warp may access: 32*quad ..
    const int row_in_item = tile * kTileRows + quad * 32 + lane;
    int ts = 0;
    uint32_t tphase = 0;
    for (int item = blockIdx.x; item < a.nitems && !*abort_flag; item += gridDim.x) {
      int b, p, sp, k0, k1;
      if (!item_range(a, item, b, p, sp, k0, k1)) continue;
      const int local = p * kItemRows + row_in_item;  // row within sequence b
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
      bool ok = true;
      for (int kb = k0; kb < k1; ++kb) {
        // warp-uniform: a timeout in any lane stops the whole warp before the
        // .sync.aligned TMEM loads
        if (!__all_sync(0xffffffffu, mbar_wait(&tm_full[ts], tphase, a.status))) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + ts * 256 + tile * 128;
        uint32_t v[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(taddr + c * 32, v[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tm_empty[ts]);
        if (++ts == 2) { ts = 0; tphase ^= 1; }
        float m[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float x = fmax3(__uint_as_float(v[c][0]), __uint_as_float(v[c][1]), __uint_as_float(v[c][2]));
#pragma unroll
          for (int e = 3; e < 31; e += 2)
            x = fmax3(x, __uint_as_float(v[c][e]), __uint_as_float(v[c][e + 1]));
          m[c] = fmaxf(x, __uint_as_float(v[c][31]));
        }
        const float mb = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
        if (valid && kb < lb && mb > sc[kCand - 1]) {
          float cs = mb;
          int ci = kb;
#pragma unroll
          for (int j = 0; j < kCand; ++j) {
            const bool better = cs > sc[j] || (cs == sc[j] && ci < id[j]);
            const float tsc = sc[j];
            const int tid = id[j];
            sc[j] = better ? cs : tsc;
            id[j] = better ? ci : tid;
            cs = better ? tsc : cs;
            ci = better ? tid : ci;
          }
        }
      }
      if (!ok) break;
      if (valid) {
        Cand* out = a.cand + ((((size_t)b * T + qi) * a.nsplit + sp) * G + g) * kCand;
#pragma unroll
        for (int j = 0; j < kCand; ++j) out[j] = Cand{sc[j], id[j]};
      }
    }
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
    cuuint64_t dims[2] = {(cuuint64_t)DI, (cuuint64_t)(s.B * cap)};
    cuuint64_t strides[1] = {(cuuint64_t)DI * 2};
    cuuint32_t box[2] = {(cuuint32_t)DI, (cuuint32_t)kBlock};
    if (!encode_bf16_map(&tm_k, k_idx, 2, dims, strides, box,
                         DI == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  IndexTcArgs a;
  a.s = s;
  a.pos = pos;
  a.npairs = (int)((s.T * (int64_t)s.G + kItemRows - 1) / kItemRows);
  a.nsplit = index_tc_nsplit(s.max_blocks);
  a.nitems = s.B * a.npairs * a.nsplit;
  a.cap = cap;
  a.cand = ws.cand;
  a.status = ws.status;
  cudaError_t e = cudaFuncSetAttribute(index_tc_kernel<DI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = a.nitems < sm_count() ? a.nitems : sm_count();
  note_launches(1);
  index_tc_kernel<DI><<<grid, kThreads, C::kSmem, st>>>(tm_q, tm_k, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_topk_merge(s, pos, 0, s.T, kSplitBlocks, a.nsplit, ws.cand, sel, st);
}

}  // namespace

size_t tc_index_workspace_bytes(const Shape& s) {
  return (size_t)s.B * s.T * index_tc_nsplit(s.max_blocks) * s.G * kCand * sizeof(Cand);
}

cudaError_t launch_index_tc(const Shape& s, const Positions& pos, const uint16_t* q_idx,
                            const uint16_t* k_idx, int32_t* sel, const Workspace& ws,
                            cudaStream_t st) {
  if (s.Di == 64) return launch_index_tc_impl<64>(s, pos, q_idx, k_idx, sel, ws, st);
  return launch_index_tc_impl<32>(s, pos, q_idx, k_idx, sel, ws, st);
}

}  // namespace msa
