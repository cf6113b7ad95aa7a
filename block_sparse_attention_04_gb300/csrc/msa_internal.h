// Internal interface between the libmsa host entry points and its kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/msa.h"

namespace msa {

constexpr int kBlock = MSA_BLOCK;     // tokens per KV block
constexpr int kTopk = MSA_TOPK;       // selected blocks per (query, group)
constexpr int kCand = MSA_TOPK - 1;   // ranked candidates besides the local block
constexpr int kMaxBatch = MSA_MAX_BATCH;
constexpr int kDevTimeout = 1;        // status word value: a bounded wait ran out
constexpr int kDevInvalid = 2;        // status word value: a selected id out of range

// Poll cap of the kernels' pipeline waits (0: the wall-clock bound alone);
// set only through msa_debug_set_wait_polls.
uint32_t debug_wait_polls();

// Adds n to the library-wide count of enqueued kernels.
void note_launches(int n);

// Per-sequence positions, passed to kernels by value (host-validated).
struct Positions {
  int32_t q_start[kMaxBatch];
  int32_t kv_len[kMaxBatch];
};

// A ranked candidate: pooled score and block id.  Order: higher score first,
// lower id on equal scores.  Empty slots hold (-inf, INT32_MAX).
struct Cand {
  float score;
  int32_t id;
};

struct Shape {
  int B, T, H, G, D, Di, max_blocks;
  float scale;
  // Paged caches: bt[B][max_blocks] maps a sequence's logical block to a block
  // of pools of pool_blocks blocks.  bt == nullptr: each sequence owns
  // max_blocks consecutive blocks (logical block kb of sequence b is block
  // b * max_blocks + kb).
  const int32_t* bt = nullptr;
  int pool_blocks = 0;
  // Blocks the cache tensors hold (the extent of their tensor maps).
  __host__ __device__ int64_t cache_blocks() const { return bt ? (int64_t)pool_blocks : (int64_t)B * max_blocks; }
};

// Scratch carved out of the caller's workspace.
struct Workspace {
  int* status;            // one status word (kDevTimeout on a wait expiry)
  int32_t* sel;           // [B][T][G][16] when the caller passes no sel buffer
  Cand* cand;             // index-scan partial candidate lists
  size_t cand_count;      // capacity of cand in entries
  float* part_o;          // attention partial outputs
  float* part_ml;         // attention partial (max, sum) pairs
  size_t part_rows;       // capacity of part_ml in (row, head, slot) entries
  char* tc_base;          // scratch of the tensor-core prefill kernels
  size_t tc_bytes;
};

// Host-side argument checks shared by every entry point (MSA_OK or a status).
int validate_params(const msa_params* p);
int validate_positions(const msa_params* p, const int32_t* q_start, const int32_t* kv_len,
                       Positions* pos);
Shape shape_of(const msa_params* p, const int32_t* block_table = nullptr, int pool_blocks = 0);

// One chunk of a dense attention call (msa_dense_attn): the chunk's selection
// holds 16 consecutive blocks; instead of writing out, the merge folds the
// chunk's block partials into running per-(query, head) accumulators (fp32
// O relative to m, in log2 units, and l), and the last chunk writes out.
struct DenseStep {
  float* acc_o;     // [B*T][H][D]
  float2* acc_ml;   // [B*T][H]
  bool first, last;
};


// ---- streaming kernels (any shape; the decode path) -----------------------
// Rows of a pass are queries [t0, t1) of every sequence.
cudaError_t launch_index_stream(const Shape& s, const Positions& pos, int t0, int t1,
                                const uint16_t* q_idx, const uint16_t* k_idx, int32_t* sel,
                                const Workspace& ws, cudaStream_t st);
size_t index_stream_cand_entries(const Shape& s, int rows, int max_lb);

// Merge of per-split candidate lists cand[(b,i)][nsplit][G][15] (split j
// covering key blocks [j*bps, (j+1)*bps)) into sel, for queries [t0, t1).
cudaError_t launch_topk_merge(const Shape& s, const Positions& pos, int t0, int t1, int bps,
                              int nsplit, const Cand* cand, int32_t* sel, cudaStream_t st);

cudaError_t launch_attn_stream(const Shape& s, const Positions& pos, int t0, int t1,
                               const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* sel, uint16_t* out, const Workspace& ws,
                               cudaStream_t st, const DenseStep* dense = nullptr);

// Dense attention: the selection of chunk j (blocks 16j .. 16j+15 that are
// causal for each query, -1 elsewhere) for every query of the call.
cudaError_t launch_dense_sel(const Shape& s, const Positions& pos, int chunk, int32_t* sel,
                             cudaStream_t st);
size_t attn_stream_part_rows(const Shape& s, int rows);

int max_local_block(const Shape& s, const Positions& pos, int t0, int t1);

// ---- cache writer --------------------------------------------------------
// Rows q_start[b] .. q_start[b] + T - 1 of every sequence, from new-token
// tensors [B][T][G][D] (K, V) and [B][T][Di] (K_idx).
cudaError_t launch_cache_append(const Shape& s, const Positions& pos, const uint16_t* k_new,
                                const uint16_t* v_new, const uint16_t* kidx_new, uint16_t* k_cache,
                                uint16_t* v_cache, uint16_t* kidx_cache, int* status,
                                cudaStream_t st);

// ---- index-branch training signal (KL(P || Q) and its gradient) ----------
size_t kl_workspace_bytes(const Shape& s);
cudaError_t launch_index_kl(const Shape& s, const Positions& pos, const uint16_t* q_idx,
                            const uint16_t* k_idx, const uint16_t* q, const uint16_t* k,
                            const int32_t* sel, float* kl, float* dq_idx, float* dk_idx, char* ws,
                            cudaStream_t st);

// ---- selection quality (evaluation of a selection against full attention) --
size_t quality_workspace_bytes(const Shape& s);
cudaError_t launch_quality(const Shape& s, const Positions& pos, const uint16_t* q,
                           const uint16_t* k, const int32_t* sel, float* coverage, float* best,
                           int32_t* dense_sel, int32_t* hits, char* ws, cudaStream_t st);

}  // namespace msa
