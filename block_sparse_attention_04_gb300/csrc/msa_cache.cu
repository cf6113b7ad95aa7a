// Cache writer: appends new tokens' K, V and K_idx rows to the block-major
// caches ("前沿架构解码手记（三）：MiniMax M2.7 → M3" section 2.1: KV laid out
// block -> token -> head -> dim, so a selected block is one contiguous run).
// With a block table the caches are pools of 128-token blocks shared by all
// sequences (vLLM-style paging at the granularity of one MSA block); without
// one, each sequence owns max_blocks consecutive blocks.
//
// One thread moves one 16-byte chunk: a token's K row (G*D bf16), V row and
// K_idx row (Di bf16) are G*D/8, G*D/8 and Di/8 chunks.  Pure data movement,
// bound by HBM: 2 * (2*G*D + Di) bytes per token.
#include "msa_device.cuh"

namespace msa {
namespace {

__global__ void __launch_bounds__(256) cache_append_kernel(
    Shape s, Positions pos, const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const uint4* __restrict__ kidx_new, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    uint4* __restrict__ kidx_cache, int* __restrict__ status) {
  const int kv_chunks = s.G * s.D / 8;      // 16-byte chunks of one token's K (or V) row
  const int ki_chunks = s.Di / 8;           // ... of its K_idx row
  const int per_tok = 2 * kv_chunks + ki_chunks;
  const int64_t n = (int64_t)s.B * s.T * per_tok;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = e / per_tok;        // (sequence, new token) = b * T + i
    const int c = (int)(e - tok * per_tok);
    const int b = (int)(tok / s.T), i = (int)(tok - (int64_t)b * s.T);
    const int64_t t = (int64_t)pos.q_start[b] + i;     // its absolute position
    const int64_t pb = cache_block(s, b, (int)(t / kBlock), status);
    if (pb < 0) continue;                   // flagged: nothing written
    const int64_t slot = pb * kBlock + (t % kBlock);   // its row in the cache
    if (c < kv_chunks) {
      k_cache[slot * kv_chunks + c] = k_new[tok * kv_chunks + c];
    } else if (c < 2 * kv_chunks) {
      v_cache[slot * kv_chunks + (c - kv_chunks)] = v_new[tok * kv_chunks + (c - kv_chunks)];
    } else {
      kidx_cache[slot * ki_chunks + (c - 2 * kv_chunks)] =
          kidx_new[tok * ki_chunks + (c - 2 * kv_chunks)];
    }
  }
}

}  // namespace

cudaError_t launch_cache_append(const Shape& s, const Positions& pos, const uint16_t* k_new,
                                const uint16_t* v_new, const uint16_t* kidx_new, uint16_t* k_cache,
                                uint16_t* v_cache, uint16_t* kidx_cache, int* status,
                                cudaStream_t st) {
  const int64_t n = (int64_t)s.B * s.T * (2 * s.G * s.D / 8 + s.Di / 8);
  if (n == 0) return cudaSuccess;
  constexpr int64_t kMaxGrid = 1 << 16;   // the kernel strides over the rest
  const int64_t blocks = (n + 255) / 256;
  note_launches(1);
  cache_append_kernel<<<(unsigned)(blocks < kMaxGrid ? blocks : kMaxGrid), 256, 0, st>>>(
      s, pos, reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<const uint4*>(kidx_new), reinterpret_cast<uint4*>(k_cache),
      reinterpret_cast<uint4*>(v_cache), reinterpret_cast<uint4*>(kidx_cache), status);
  return cudaGetLastError();
}

}  // namespace msa
