// Synthetic-input generator (benchmarks and tests only; none of the
// attention or allocation method).  Same definition as the numpy generator:
// SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014) over a
// counter, four 16-bit fields summed and scaled to ~N(0, 1) in float32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "swa_synth.h"

namespace {

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void k_synth(uint64_t base, int32_t layer, const int64_t *req, const int64_t *pos,
                        int64_t n, int32_t heads, int32_t dim, int32_t bf16, void *out) {
  const int64_t total = n * heads * dim;
  const float scale = 0x1.bb67aep-16f;  // float32(sqrt(3) / 65536)
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    int64_t i = e / ((int64_t)heads * dim);
    int64_t r = e % ((int64_t)heads * dim);
    uint64_t h = (uint64_t)(r / dim), d = (uint64_t)(r % dim);
    uint64_t idx = ((uint64_t)layer << 47) | ((uint64_t)req[i] << 35) |
                   ((uint64_t)pos[i] << 15) | (h << 8) | d;
    uint64_t z = mix64(base + (idx + 1ull) * 0x9E3779B97F4A7C15ull);
    int64_t sum = (int64_t)(z & 0xFFFF) + (int64_t)((z >> 16) & 0xFFFF) +
                  (int64_t)((z >> 32) & 0xFFFF) + (int64_t)(z >> 48);
    float x = __fmul_rn((float)(sum - 131070), scale);
    if (bf16) static_cast<__nv_bfloat16 *>(out)[e] = __float2bfloat16_rn(x);
    else static_cast<float *>(out)[e] = x;
  }
}

}  // namespace

extern "C" swa_status swa_synth_tokens(uint64_t seed, int32_t stream_id, int32_t layer,
                                       const int64_t *req, const int64_t *pos, int64_t n,
                                       int32_t heads, int32_t dim, int32_t out_dtype, void *out,
                                       swa_stream_t stream) {
  if (n < 0 || heads <= 0 || dim <= 0 || (n > 0 && (!req || !pos || !out))) return SWA_ERR_INVALID;
  if (n == 0) return SWA_OK;
  uint64_t base = mix64((seed << 32) ^ (uint64_t)(uint32_t)stream_id);
  int64_t total = n * heads * dim;
  int64_t grid = (total + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  k_synth<<<(int)grid, 256, 0, (cudaStream_t)stream>>>(base, layer, req, pos, n, heads, dim,
                                                       out_dtype != SWA_DTYPE_F32, out);
  return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}
