// Tensor-core (tcgen05) prefill kernels of libmsa.
#pragma once
#include "msa_internal.h"

namespace msa {

// Bytes of scratch the tensor-core index scan and KV-outer attention need.
size_t tc_workspace_bytes(const Shape& s);

// Steps 1-3 for every query of the call (tcgen05 index scan + merge).
cudaError_t launch_index_tc(const Shape& s, const Positions& pos, const uint16_t* q_idx,
                            const uint16_t* k_idx, int32_t* sel, const Workspace& ws,
                            cudaStream_t st);

// Step 4 for every query of the call (KV-outer tcgen05 attention + merge).
cudaError_t launch_attn_tc(const Shape& s, const Positions& pos, const uint16_t* q,
                           const uint16_t* k, const uint16_t* v, const int32_t* sel,
                           uint16_t* out, const Workspace& ws, cudaStream_t st);

}  // namespace msa
