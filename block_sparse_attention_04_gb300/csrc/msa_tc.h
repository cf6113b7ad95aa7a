// Tensor-core (tcgen05) prefill kernels of libmsa.
#pragma once
#include "msa_internal.h"

namespace msa {

// Scratch bytes of the tensor-core index scan: per-split candidate lists of
// every (query, group) of the call.
size_t tc_index_workspace_bytes(const Shape& s);

// Steps 1-3 for every query of the call (tcgen05 index scan + merge).
cudaError_t launch_index_tc(const Shape& s, const Positions& pos, const uint16_t* q_idx,
                            const uint16_t* k_idx, int32_t* sel, const Workspace& ws,
                            cudaStream_t st);

// Queries per sequence in one pass of the tensor-core attention (the pass
// bounds its scratch: at most 8192 (sequence, query) rows).
int pass_len(const Shape& s);

// Scratch bytes of the KV-outer attention for one pass.
size_t tc_attn_workspace_bytes(const Shape& s);

// Step 4 for every query of the call (inverted lists, KV-outer tcgen05
// attention, log-sum-exp merge), in passes of pass_len(s) queries.
cudaError_t launch_attn_tc(const Shape& s, const Positions& pos, const uint16_t* q,
                           const uint16_t* k, const uint16_t* v, const int32_t* sel,
                           uint16_t* out, const Workspace& ws, cudaStream_t st);

// Dense causal attention of every query of the call over all its causal
// keys (query-outer tcgen05 kernel, O kept in tensor memory).
cudaError_t launch_dense_tc(const Shape& s, const Positions& pos, const uint16_t* q,
                            const uint16_t* k, const uint16_t* v, uint16_t* out, int* status,
                            cudaStream_t st);

}  // namespace msa
