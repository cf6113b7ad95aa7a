// Tensor-core prefill kernels: not built yet; the host entry points reject a
// request for them with MSA_ERR_UNSUPPORTED.
#include "msa_tc.h"

namespace msa {

size_t tc_workspace_bytes(const Shape&) { return 0; }

cudaError_t launch_index_tc(const Shape&, const Positions&, const uint16_t*, const uint16_t*,
                            int32_t*, const Workspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_attn_tc(const Shape&, const Positions&, const uint16_t*, const uint16_t*,
                           const uint16_t*, const int32_t*, uint16_t*, const Workspace&,
                           cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace msa
