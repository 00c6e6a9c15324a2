// E4M3 encoding of stored K/V ("SGLang source teardown (15)", section "second
// mapping: the KV store": FP8 pools hold raw bytes): each value is divided by
// the per-tensor scale in float32 (round to nearest) and converted with
// round-to-nearest-even and saturation to +-448.  Shared by every kernel that
// writes pool rows, so all of them produce the same bytes.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace swa {

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// 16 output bytes from 16 bf16 inputs (two 16-byte words).
__device__ __forceinline__ uint4 e4m3_encode16(uint4 a, uint4 b, float scale) {
  const __nv_bfloat16 *ha = reinterpret_cast<const __nv_bfloat16 *>(&a);
  const __nv_bfloat16 *hb = reinterpret_cast<const __nv_bfloat16 *>(&b);
  float f[16];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    f[e] = __fdiv_rn(__bfloat162float(ha[e]), scale);
    f[8 + e] = __fdiv_rn(__bfloat162float(hb[e]), scale);
  }
  uint4 o;
  o.x = pack_e4m3x4(f[0], f[1], f[2], f[3]);
  o.y = pack_e4m3x4(f[4], f[5], f[6], f[7]);
  o.z = pack_e4m3x4(f[8], f[9], f[10], f[11]);
  o.w = pack_e4m3x4(f[12], f[13], f[14], f[15]);
  return o;
}

}  // namespace swa
