// msa_index_topk_noalloc: the streaming index scan (score, pool, top-16 with
// the local block forced) for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a serving engine that hands
// every free byte of the GPU to its KV-cache pool at start-up and forbids
// allocations afterwards, or a plugin host that only passes the library its
// input and output buffers.  They cannot provide the workspace that
// msa_index_topk needs either.  This entry point keeps its scratch (the
// per-split candidate lists) in a file-scope __device__ array instead, so it
// allocates nothing and needs no workspace argument.
#include <mutex>

#include "msa_internal.h"

namespace msa {
namespace {

// The scratch: MSA_NOALLOC_SCRATCH_BYTES bytes of device memory that every GPU
// on which this library's module is loaded holds until the process exits.
// In host code this name is only a host-side stand-in for the symbol, never a
// device address; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Set-up, once per device, with that device current: look up the device
// address of the scratch array.  The first call on each device does this.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
      return MSA_ERR_CUDA;
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" int msa_index_topk_noalloc(const msa_params* p, const uint16_t* q_idx,
                                      const uint16_t* k_idx, const int32_t* q_start,
                                      const int32_t* kv_len, int32_t* sel, cudaStream_t stream) {
  int rc = validate_params(p);
  if (rc) return rc;
  Positions pos;
  if ((rc = validate_positions(p, q_start, kv_len, &pos))) return rc;
  if (!q_idx || !k_idx || !sel) return MSA_ERR_INVALID_ARG;
  if (((uintptr_t)q_idx | (uintptr_t)k_idx | (uintptr_t)sel) & 15u) return MSA_ERR_INVALID_ARG;
  if (p->T == 0) return MSA_OK;
  if ((int64_t)p->B * p->T > 65535) return MSA_ERR_UNSUPPORTED;  // one launch covers all rows
  const Shape s = shape_of(p);
  const int max_lb = max_local_block(s, pos, 0, p->T);
  const size_t need = index_stream_cand_entries(s, p->B * p->T, max_lb) * sizeof(Cand);
  if (need > (size_t)MSA_NOALLOC_SCRATCH_BYTES) return MSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch))) return rc;
  // Every candidate entry the merge reads is written earlier in the same
  // call, so the previous call's contents need no clearing.
  Workspace w{};
  w.cand = static_cast<Cand*>(scratch);
  w.cand_count = need / sizeof(Cand);
  return launch_index_stream(s, pos, 0, p->T, q_idx, k_idx, sel, w, stream) == cudaSuccess
             ? MSA_OK
             : MSA_ERR_CUDA;
}
