// Device-side fill of the seeded synthetic inputs defined in msa_synth/__init__.py
// (SplitMix64 counter hash; Irwin-Hall "normal" and 2^-3 "grid" values; K_idx
// needles).  Holds no attention arithmetic.  Each function fills one tensor of
// one sequence on the given stream and returns a cudaError_t as int.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t stream_key(uint64_t seed, int tid, int b) {
  uint64_t k = mix64(seed + kGamma * (uint64_t)(tid + 1));
  return mix64(k + kGamma * (uint64_t)(b + 1));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float x) {
  uint32_t u = __float_as_uint(x);
  u += ((u >> 16) & 1u) + 0x7FFFu;
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ uint16_t normal_bits(uint64_t h) {
  uint32_t s = (uint32_t)(h & 0xFFFF) + (uint32_t)((h >> 16) & 0xFFFF) + (uint32_t)((h >> 32) & 0xFFFF);
  int32_t v = 2 * (int32_t)s - 196605;
  return f32_to_bf16_rne((float)v * 1.52587890625e-05f);  // 2^-16, exact
}

__device__ __forceinline__ uint16_t grid_bits(uint64_t h) {
  int k = (int)(h % 17ull) - 8;
  return f32_to_bf16_rne((float)k * 0.125f);
}

template <bool kNormal>
__global__ void fill_kernel(uint16_t* __restrict__ out, int64_t n, uint64_t key, int64_t idx0) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
  for (int64_t base = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; base < n; base += stride) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int64_t k = base + e;
      if (k < n) {
        uint64_t h = mix64(key + kGamma * (uint64_t)(idx0 + k + 1));
        out[k] = kNormal ? normal_bits(h) : grid_bits(h);
      }
    }
  }
}

__global__ void needle_kernel(uint16_t* __restrict__ kidx, int64_t nneedle, int di,
                              uint64_t key_tok, uint64_t key_dim) {
  int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= nneedle) return;
  uint64_t n = (uint64_t)j + 4;          // needle ids start at 4*qb with qb = 1
  uint64_t qb = n / 4;
  uint64_t tok = mix64(key_tok + kGamma * (n + 1)) % (qb * 128ull);
  for (int m = 0; m < 8; ++m) {
    uint64_t d = mix64(key_dim + kGamma * (n * 8ull + (uint64_t)m + 1)) % (uint64_t)di;
    kidx[tok * (uint64_t)di + d] = 0x4080;  // bf16 bits of 4.0
  }
}

int grid_for(int64_t n) {
  int64_t g = (n / 4 + 255) / 256;
  if (g < 1) g = 1;
  if (g > 65536) g = 65536;
  return (int)g;
}

}  // namespace

extern "C" {

// out[k] = normal(h(seed, tid, b, idx0 + k)), k in [0, n)
int msa_synth_normal(uint16_t* out, int64_t n, uint64_t seed, int tid, int b, int64_t idx0,
                     cudaStream_t stream) {
  if (n <= 0) return 0;
  fill_kernel<true><<<grid_for(n), 256, 0, stream>>>(out, n, stream_key(seed, tid, b), idx0);
  return (int)cudaGetLastError();
}

// out[k] = grid(h(seed, tid, b, idx0 + k)), k in [0, n)
int msa_synth_grid(uint16_t* out, int64_t n, uint64_t seed, int tid, int b, int64_t idx0,
                   cudaStream_t stream) {
  if (n <= 0) return 0;
  fill_kernel<false><<<grid_for(n), 256, 0, stream>>>(out, n, stream_key(seed, tid, b), idx0);
  return (int)cudaGetLastError();
}

// Plant the needles of sequence b (whole context ctx_len tokens) into its K_idx
// rows kidx[tok][di] (the caller's buffer holds at least ctx_len rows).
int msa_synth_needles(uint16_t* kidx, int64_t ctx_len, int di, uint64_t seed, int b,
                      cudaStream_t stream) {
  int64_t nb = (ctx_len + 127) / 128;
  if (nb < 2) return 0;
  int64_t nneedle = (nb - 1) * 4;
  int grid = (int)((nneedle + 255) / 256);
  needle_kernel<<<grid, 256, 0, stream>>>(kidx, nneedle, di, stream_key(seed, 6, b),
                                          stream_key(seed, 7, b));
  return (int)cudaGetLastError();
}

}  // extern "C"
