// libmsa C ABI (include/msa.h): argument validation, workspace layout and the
// launch sequence of the MSA forward pass.  All arithmetic runs in the
// kernels; this file only checks arguments, carves the caller's workspace and
// enqueues launches on the caller's stream.
#include <atomic>
#include <cmath>
#include <cstring>

#include "msa_internal.h"
#include "msa_tc.h"

namespace msa {

static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static std::atomic<uint32_t> g_wait_polls{0};
uint32_t debug_wait_polls() { return g_wait_polls.load(std::memory_order_relaxed); }

constexpr int kMaxContextBlocks = 32768;

int validate_params(const msa_params* p) {
  if (!p) return MSA_ERR_INVALID_ARG;
  if (p->B < 1 || p->T < 0 || p->H < 1 || p->G < 1 || p->max_blocks < 1)
    return MSA_ERR_INVALID_ARG;
  if (p->H % p->G != 0) return MSA_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale)) return MSA_ERR_INVALID_ARG;
  if (p->kernels < MSA_KERNELS_AUTO || p->kernels > MSA_KERNELS_TENSORCORE)
    return MSA_ERR_INVALID_ARG;
  if (p->B > MSA_MAX_BATCH) return MSA_ERR_UNSUPPORTED;
  if (p->block != MSA_BLOCK || p->topk != MSA_TOPK) return MSA_ERR_UNSUPPORTED;
  if (p->D != 64 && p->D != 128) return MSA_ERR_UNSUPPORTED;
  if (p->Di != 32 && p->Di != 64) return MSA_ERR_UNSUPPORTED;
  if (p->G > 8 || p->H / p->G > 16) return MSA_ERR_UNSUPPORTED;
  if (p->max_blocks > kMaxContextBlocks) return MSA_ERR_UNSUPPORTED;
  // TMA coordinates are 32-bit: rows of q_idx, q (one per head) and k_idx must fit
  if ((int64_t)p->B * p->T * p->G >= ((int64_t)1 << 31) ||
      (int64_t)p->B * p->T * p->H >= ((int64_t)1 << 31) ||
      (int64_t)p->B * p->max_blocks * MSA_BLOCK >= ((int64_t)1 << 31))
    return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

int validate_positions(const msa_params* p, const int32_t* q_start, const int32_t* kv_len,
                       Positions* pos) {
  if (!q_start || !kv_len) return MSA_ERR_INVALID_ARG;
  std::memset(pos, 0, sizeof(*pos));
  const int64_t cap = (int64_t)p->max_blocks * MSA_BLOCK;
  for (int b = 0; b < p->B; ++b) {
    if (q_start[b] < 0 || kv_len[b] < 0) return MSA_ERR_INVALID_ARG;
    if ((int64_t)q_start[b] + p->T > kv_len[b]) return MSA_ERR_INVALID_ARG;
    if ((int64_t)kv_len[b] > cap) return MSA_ERR_INVALID_ARG;
    pos->q_start[b] = q_start[b];
    pos->kv_len[b] = kv_len[b];
  }
  return MSA_OK;
}

Shape shape_of(const msa_params* p, const int32_t* block_table, int pool_blocks) {
  Shape s{p->B, p->T, p->H, p->G, p->D, p->Di, p->max_blocks, p->scale};
  s.bt = block_table;
  s.pool_blocks = pool_blocks;
  return s;
}


namespace {

constexpr size_t kAlign = 256;
constexpr int kStreamRows = 2048;   // query rows per streaming pass

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Index scan on tensor cores for prefill-sized calls (>= 256 query-group rows
// per sequence fill one work item), streaming otherwise.
bool use_tc_index(const msa_params* p) {
  if (p->kernels == MSA_KERNELS_TENSORCORE) return true;
  if (p->kernels == MSA_KERNELS_STREAMING) return false;
  return (int64_t)p->T * p->G >= 256;
}

// KV-outer tensor-core attention for prefill-sized calls.
bool use_tc_attn(const msa_params* p) { return use_tc_index(p); }

int stream_pass_len(const msa_params* p) {
  int tc = kStreamRows / p->B;
  if (tc < 1) tc = 1;
  return tc < p->T ? tc : (p->T > 0 ? p->T : 1);
}

struct Plan {
  size_t status_off, sel_off, scratch_off, total;
  size_t cand_entries, part_rows;
};

Plan plan_for(const msa_params* p) {
  Plan pl{};
  const Shape s = shape_of(p);
  const int max_lb = p->max_blocks - 1;
  const int rows = p->B * stream_pass_len(p);
  size_t idx = 0, att = 0;
  if (use_tc_index(p)) {
    idx = align_up(tc_index_workspace_bytes(s));
    pl.cand_entries = idx / sizeof(Cand);
  } else {
    pl.cand_entries = index_stream_cand_entries(s, rows, max_lb);
    idx = align_up(pl.cand_entries * sizeof(Cand));
  }
  if (use_tc_attn(p)) {
    att = align_up(tc_attn_workspace_bytes(s));
  } else {
    pl.part_rows = attn_stream_part_rows(s, rows);
    att = align_up(pl.part_rows * p->D * sizeof(float)) + align_up(pl.part_rows * 2 * sizeof(float));
  }
  const size_t scratch = idx > att ? idx : att;
  pl.status_off = 0;
  pl.sel_off = kAlign;
  pl.scratch_off = pl.sel_off + align_up((size_t)p->B * p->T * p->G * MSA_TOPK * sizeof(int32_t));
  pl.total = pl.scratch_off + scratch;
  return pl;
}

Workspace carve(const msa_params* p, const Plan& pl, void* ws) {
  char* base = static_cast<char*>(ws);
  Workspace w{};
  w.status = reinterpret_cast<int*>(base + pl.status_off);
  w.sel = reinterpret_cast<int32_t*>(base + pl.sel_off);
  char* scr = base + pl.scratch_off;
  w.cand = reinterpret_cast<Cand*>(scr);
  w.cand_count = pl.cand_entries;
  w.part_o = reinterpret_cast<float*>(scr);
  w.part_rows = pl.part_rows;
  w.part_ml = reinterpret_cast<float*>(scr + align_up(pl.part_rows * p->D * sizeof(float)));
  w.tc_base = scr;
  w.tc_bytes = pl.total - pl.scratch_off;
  return w;
}

int check_ws(const msa_params* p, void* ws, size_t ws_bytes, Plan* pl) {
  if (!ws || ((uintptr_t)ws & (kAlign - 1)) != 0) return MSA_ERR_INVALID_ARG;
  *pl = plan_for(p);
  if (ws_bytes < pl->total) return MSA_ERR_WORKSPACE;
  return MSA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

int run_index(const msa_params* p, const Shape& s, const Positions& pos, const uint16_t* q_idx,
              const uint16_t* k_idx, int32_t* sel, const Workspace& w, cudaStream_t st) {
  if (use_tc_index(p)) return cuda_status(launch_index_tc(s, pos, q_idx, k_idx, sel, w, st));
  const int tc = stream_pass_len(p);
  for (int t0 = 0; t0 < p->T; t0 += tc) {
    const int t1 = t0 + tc < p->T ? t0 + tc : p->T;
    cudaError_t e = launch_index_stream(s, pos, t0, t1, q_idx, k_idx, sel, w, st);
    if (e != cudaSuccess) return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

int run_attn(const msa_params* p, const Shape& s, const Positions& pos, const uint16_t* q,
             const uint16_t* k, const uint16_t* v, const int32_t* sel, uint16_t* out,
             const Workspace& w, cudaStream_t st) {
  if (use_tc_attn(p)) return cuda_status(launch_attn_tc(s, pos, q, k, v, sel, out, w, st));
  const int tc = stream_pass_len(p);
  for (int t0 = 0; t0 < p->T; t0 += tc) {
    const int t1 = t0 + tc < p->T ? t0 + tc : p->T;
    cudaError_t e = launch_attn_stream(s, pos, t0, t1, q, k, v, sel, out, w, st);
    if (e != cudaSuccess) return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

// Workspace of msa_dense_attn.  Tensor-core shapes: the status word only
// (one query-outer kernel keeps everything else on chip).  Streaming shapes:
// status word, the chunk selection, the running accumulators, then the
// streaming attention's scratch.
struct DensePlan {
  size_t sel_off, acc_o_off, acc_ml_off, scratch_off, total, part_rows;
};

DensePlan dense_plan_for(const msa_params* p) {
  DensePlan d{};
  if (use_tc_attn(p)) {
    d.total = kAlign;
    return d;
  }
  const Shape s = shape_of(p);
  const size_t rows = (size_t)p->B * p->T;
  d.part_rows = attn_stream_part_rows(s, p->B * stream_pass_len(p));
  const size_t att =
      align_up(d.part_rows * p->D * sizeof(float)) + align_up(d.part_rows * 2 * sizeof(float));
  d.sel_off = kAlign;
  d.acc_o_off = d.sel_off + align_up(rows * p->G * MSA_TOPK * sizeof(int32_t));
  d.acc_ml_off = d.acc_o_off + align_up(rows * p->H * p->D * sizeof(float));
  d.scratch_off = d.acc_ml_off + align_up(rows * p->H * 2 * sizeof(float));
  d.total = d.scratch_off + att;
  return d;
}

// A pool of num_pool_blocks 128-token blocks: its rows (tensor-copy
// coordinates) must fit 32 bits, like those of per-sequence caches.
int validate_pool(const int32_t* block_table, int num_pool_blocks) {
  if (!block_table || num_pool_blocks < 1) return MSA_ERR_INVALID_ARG;
  if (((uintptr_t)block_table & 3u) != 0) return MSA_ERR_INVALID_ARG;
  if ((int64_t)num_pool_blocks * MSA_BLOCK + MSA_BLOCK >= ((int64_t)1 << 31))
    return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

// Steps 1-4 for msa_forward and msa_forward_paged (s carries the block table,
// or none); p is validated.
int forward(const msa_params* p, const Shape& s, const uint16_t* q_idx, const uint16_t* k_idx,
            const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
            const int32_t* q_start, const int32_t* kv_len, int32_t* sel_out, uint16_t* out,
            void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc;
  Positions pos;
  if ((rc = validate_positions(p, q_start, kv_len, &pos))) return rc;
  if (!q_idx || !k_idx || !q || !k_cache || !v_cache || !out) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(q) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (sel_out && !aligned16(sel_out)))
    return MSA_ERR_INVALID_ARG;
  Plan pl;
  if ((rc = check_ws(p, ws, ws_bytes, &pl))) return rc;
  if (p->T == 0) return MSA_OK;
  Workspace w = carve(p, pl, ws);
  int32_t* sel = sel_out ? sel_out : w.sel;
  if (cudaMemsetAsync(w.status, 0, sizeof(int), stream) != cudaSuccess) return MSA_ERR_CUDA;
  if ((rc = run_index(p, s, pos, q_idx, k_idx, sel, w, stream))) return rc;
  return run_attn(p, s, pos, q, k_cache, v_cache, sel, out, w, stream);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_workspace_bytes(const msa_params* p) {
  if (validate_params(p) != MSA_OK) return 0;
  return plan_for(p).total;
}

int msa_index_topk(const msa_params* p, const uint16_t* q_idx, const uint16_t* k_idx,
                   const int32_t* q_start, const int32_t* kv_len, int32_t* sel, void* ws,
                   size_t ws_bytes, cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  Positions pos;
  if ((rc = validate_positions(p, q_start, kv_len, &pos))) return rc;
  if (!q_idx || !k_idx || !sel) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(sel)) return MSA_ERR_INVALID_ARG;
  Plan pl;
  if ((rc = check_ws(p, ws, ws_bytes, &pl))) return rc;
  if (p->T == 0) return MSA_OK;
  Workspace w = carve(p, pl, ws);
  if (cudaMemsetAsync(w.status, 0, sizeof(int), stream) != cudaSuccess) return MSA_ERR_CUDA;
  return run_index(p, shape_of(p), pos, q_idx, k_idx, sel, w, stream);
}

int msa_sparse_attn(const msa_params* p, const uint16_t* q, const uint16_t* k_cache,
                    const uint16_t* v_cache, const int32_t* sel, const int32_t* q_start,
                    const int32_t* kv_len, uint16_t* out, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  Positions pos;
  if ((rc = validate_positions(p, q_start, kv_len, &pos))) return rc;
  if (!q || !k_cache || !v_cache || !sel || !out) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(sel) ||
      !aligned16(out))
    return MSA_ERR_INVALID_ARG;
  Plan pl;
  if ((rc = check_ws(p, ws, ws_bytes, &pl))) return rc;
  if (p->T == 0) return MSA_OK;
  Workspace w = carve(p, pl, ws);
  if (cudaMemsetAsync(w.status, 0, sizeof(int), stream) != cudaSuccess) return MSA_ERR_CUDA;
  return run_attn(p, shape_of(p), pos, q, k_cache, v_cache, sel, out, w, stream);
}

int msa_forward(const msa_params* p, const uint16_t* q_idx, const uint16_t* k_idx,
                const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                const int32_t* q_start, const int32_t* kv_len, int32_t* sel_out, uint16_t* out,
                void* ws, size_t ws_bytes, cudaStream_t stream) {
  const int rc = validate_params(p);
  if (rc) return rc;
  return forward(p, shape_of(p), q_idx, k_idx, q, k_cache, v_cache, q_start, kv_len, sel_out,
                 out, ws, ws_bytes, stream);
}

int msa_forward_paged(const msa_params* p, const int32_t* block_table, int num_pool_blocks,
                      const uint16_t* q_idx, const uint16_t* k_idx_pool, const uint16_t* q,
                      const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* q_start,
                      const int32_t* kv_len, int32_t* sel_out, uint16_t* out, void* ws,
                      size_t ws_bytes, cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  if ((rc = validate_pool(block_table, num_pool_blocks))) return rc;
  return forward(p, shape_of(p, block_table, num_pool_blocks), q_idx, k_idx_pool, q, k_pool,
                 v_pool, q_start, kv_len, sel_out, out, ws, ws_bytes, stream);
}

int msa_cache_append(const msa_params* p, const int32_t* block_table, int num_pool_blocks,
                     const uint16_t* k_new, const uint16_t* v_new, const uint16_t* k_idx_new,
                     const int32_t* q_start, uint16_t* k_cache, uint16_t* v_cache,
                     uint16_t* k_idx_cache, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  if (block_table && (rc = validate_pool(block_table, num_pool_blocks))) return rc;
  if (!q_start) return MSA_ERR_INVALID_ARG;
  Positions pos;
  std::memset(&pos, 0, sizeof(pos));
  const int64_t cap = (int64_t)p->max_blocks * MSA_BLOCK;
  for (int b = 0; b < p->B; ++b) {
    if (q_start[b] < 0 || (int64_t)q_start[b] + p->T > cap) return MSA_ERR_INVALID_ARG;
    pos.q_start[b] = q_start[b];
    pos.kv_len[b] = q_start[b] + p->T;
  }
  if (!k_new || !v_new || !k_idx_new || !k_cache || !v_cache || !k_idx_cache)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_idx_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(k_idx_cache))
    return MSA_ERR_INVALID_ARG;
  if (!ws || ((uintptr_t)ws & (kAlign - 1)) != 0) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < kAlign) return MSA_ERR_WORKSPACE;
  if (p->T == 0) return MSA_OK;
  int* status = static_cast<int*>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess) return MSA_ERR_CUDA;
  return cuda_status(launch_cache_append(shape_of(p, block_table, num_pool_blocks), pos, k_new,
                                         v_new, k_idx_new, k_cache, v_cache, k_idx_cache, status,
                                         stream));
}

size_t msa_dense_workspace_bytes(const msa_params* p) {
  if (validate_params(p) != MSA_OK) return 0;
  return dense_plan_for(p).total;
}

int msa_dense_attn(const msa_params* p, const uint16_t* q, const uint16_t* k_cache,
                   const uint16_t* v_cache, const int32_t* q_start, const int32_t* kv_len,
                   uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  Positions pos;
  if ((rc = validate_positions(p, q_start, kv_len, &pos))) return rc;
  if (!q || !k_cache || !v_cache || !out) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return MSA_ERR_INVALID_ARG;
  if (!ws || ((uintptr_t)ws & (kAlign - 1)) != 0) return MSA_ERR_INVALID_ARG;
  const DensePlan d = dense_plan_for(p);
  if (ws_bytes < d.total) return MSA_ERR_WORKSPACE;
  if (p->T == 0) return MSA_OK;
  char* base = static_cast<char*>(ws);
  Workspace w{};
  w.status = reinterpret_cast<int*>(base);
  int32_t* sel = reinterpret_cast<int32_t*>(base + d.sel_off);
  char* scr = base + d.scratch_off;
  w.part_o = reinterpret_cast<float*>(scr);
  w.part_rows = d.part_rows;
  w.part_ml = reinterpret_cast<float*>(scr + align_up(d.part_rows * p->D * sizeof(float)));
  w.tc_base = scr;
  w.tc_bytes = d.total - d.scratch_off;
  if (cudaMemsetAsync(w.status, 0, sizeof(int), stream) != cudaSuccess) return MSA_ERR_CUDA;
  const Shape s = shape_of(p);
  if (use_tc_attn(p))
    return cuda_status(launch_dense_tc(s, pos, q, k_cache, v_cache, out, w.status, stream));
  // streaming shapes: chunks of 16 consecutive blocks, up to the last query's
  // local block, each folded into fp32 running accumulators
  const int nchunks = (max_local_block(s, pos, 0, p->T) + MSA_TOPK) / MSA_TOPK;
  for (int c = 0; c < nchunks; ++c) {
    if (launch_dense_sel(s, pos, c, sel, stream) != cudaSuccess) return MSA_ERR_CUDA;
    DenseStep ds{reinterpret_cast<float*>(base + d.acc_o_off),
                 reinterpret_cast<float2*>(base + d.acc_ml_off), c == 0, c == nchunks - 1};
    const int tc = stream_pass_len(p);
    for (int t0 = 0; t0 < p->T; t0 += tc) {
      const int t1 = t0 + tc < p->T ? t0 + tc : p->T;
      if (launch_attn_stream(s, pos, t0, t1, q, k_cache, v_cache, sel, out, w, stream, &ds) !=
          cudaSuccess)
        return MSA_ERR_CUDA;
    }
  }
  return MSA_OK;
}

size_t msa_index_kl_workspace_bytes(const msa_params* p) {
  if (validate_params(p) != MSA_OK) return 0;
  return kl_workspace_bytes(shape_of(p));
}

int msa_index_kl(const msa_params* p, const uint16_t* q_idx, const uint16_t* k_idx,
                 const uint16_t* q, const uint16_t* k_cache, const int32_t* sel,
                 const int32_t* q_start, const int32_t* kv_len, float* kl, float* dq_idx,
                 float* dk_idx, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  Positions pos;
  if ((rc = validate_positions(p, q_start, kv_len, &pos))) return rc;
  if (!q_idx || !k_idx || !q || !k_cache || !sel || !kl || !dq_idx || !dk_idx)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(q) || !aligned16(k_cache) ||
      !aligned16(sel) || !aligned16(kl) || !aligned16(dq_idx) || !aligned16(dk_idx))
    return MSA_ERR_INVALID_ARG;
  if (!ws || ((uintptr_t)ws & (kAlign - 1)) != 0) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < kl_workspace_bytes(shape_of(p))) return MSA_ERR_WORKSPACE;
  if (p->T == 0) return MSA_OK;
  return cuda_status(launch_index_kl(shape_of(p), pos, q_idx, k_idx, q, k_cache, sel, kl, dq_idx,
                                     dk_idx, static_cast<char*>(ws), stream));
}

size_t msa_quality_workspace_bytes(const msa_params* p) {
  if (validate_params(p) != MSA_OK) return 0;
  return quality_workspace_bytes(shape_of(p));
}

int msa_selection_quality(const msa_params* p, const uint16_t* q, const uint16_t* k_cache,
                          const int32_t* sel, const int32_t* q_start, const int32_t* kv_len,
                          float* coverage, float* best_coverage, int32_t* dense_sel,
                          int32_t* hits, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  Positions pos;
  if ((rc = validate_positions(p, q_start, kv_len, &pos))) return rc;
  if (!q || !k_cache || !sel || !coverage || !best_coverage || !dense_sel || !hits)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(sel) || !aligned16(coverage) ||
      !aligned16(best_coverage) || !aligned16(dense_sel) || !aligned16(hits))
    return MSA_ERR_INVALID_ARG;
  if (!ws || ((uintptr_t)ws & (kAlign - 1)) != 0) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < quality_workspace_bytes(shape_of(p))) return MSA_ERR_WORKSPACE;
  if (p->T == 0) return MSA_OK;
  return cuda_status(launch_quality(shape_of(p), pos, q, k_cache, sel, coverage, best_coverage,
                                    dense_sel, hits, static_cast<char*>(ws), stream));
}

int msa_workspace_status(const void* ws, cudaStream_t stream) {
  if (!ws) return MSA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
  if (v == kDevTimeout) return MSA_ERR_TIMEOUT;
  if (v == kDevInvalid) return MSA_ERR_INVALID_ARG;
  return v == 0 ? MSA_OK : MSA_ERR_CUDA;
}

uint64_t msa_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void msa_debug_set_wait_polls(uint32_t polls) {
  g_wait_polls.store(polls, std::memory_order_relaxed);
}

const char* msa_status_string(int status) {
  switch (status) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported shape";
    case MSA_ERR_WORKSPACE: return "workspace too small";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_TIMEOUT: return "kernel wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
