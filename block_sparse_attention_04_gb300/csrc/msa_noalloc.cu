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
#include <cuda.h>

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

// The array's device address, looked up once per device and remembered with
// the id of the context it was looked up in.  The module (and so the array)
// belongs to a context: after cudaDeviceReset, or under another context on
// the same device, the id differs and the address is looked up again.
struct ScratchSlot {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_setup_mu;
ScratchSlot g_slots[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// The driver's context calls, looked up through the runtime (libmsa does not
// link the driver library directly).
bool driver_ctx_calls(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  static CtxGetCurrentFn f_cur = nullptr;
  static CtxGetIdFn f_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  *cur = f_cur;
  *id = f_id;
  return f_cur && f_id;
}

// Id of the calling thread's current context, 0 if there is none yet.
int current_ctx_id(unsigned long long* out) {
  CtxGetCurrentFn cur;
  CtxGetIdFn id;
  if (!driver_ctx_calls(&cur, &id)) return MSA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (cur(&ctx) != CUDA_SUCCESS) return MSA_ERR_CUDA;
  *out = 0;
  if (ctx && id(ctx, out) != CUDA_SUCCESS) return MSA_ERR_CUDA;
  return MSA_OK;
}

// Set-up, once per device (and again if that device's context changed), with
// that device current: look up the device address of the scratch array.  The
// first call on each device does this.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MSA_ERR_UNSUPPORTED;
  unsigned long long ctx = 0;
  int rc = current_ctx_id(&ctx);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  ScratchSlot& slot = g_slots[dev];
  if (ctx == 0 || slot.addr == nullptr || slot.ctx_id != ctx) {
    void* addr = nullptr;
    // makes the device's primary context current if the thread had none
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
      return MSA_ERR_CUDA;
    if ((rc = current_ctx_id(&ctx))) return rc;
    slot.ctx_id = ctx;
    slot.addr = addr;
  }
  *out = slot.addr;
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
