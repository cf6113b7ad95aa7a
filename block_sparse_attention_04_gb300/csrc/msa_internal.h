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
Shape shape_of(const msa_params* p);

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
                               cudaStream_t st);
size_t attn_stream_part_rows(const Shape& s, int rows);

int max_local_block(const Shape& s, const Positions& pos, int t0, int t1);

}  // namespace msa
