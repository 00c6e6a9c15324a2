// swa_attn_decode_noalloc: decode attention whose split-KV scratch lives in a
// fixed array inside this library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at all: serving engines that
// hand every byte of HBM to their KV pools at start-up and forbid later
// allocations, plug-ins running inside a host framework that exposes no
// allocator to them, and code paths where a cudaMalloc (which can
// synchronise the device) is not acceptable.  They still pass their inputs
// and outputs; the partial softmax results and merge tickets go to
// `g_decode_scratch` below.
//
// The array is kNoAllocScratchBytes (32 MiB) of device memory that every GPU
// loading this library keeps until the process exits.  Every call on a
// device shares it and it keeps the last call's contents, so each call
// clears the part that must start at zero (the work counters and merge
// tickets; the kernels write every partial before they read it), and calls
// that overlap on the GPU (for example on two streams) race on it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "swa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, never a device address.  The
// lookup is a host-side query that allocates nothing; it runs on every call,
// so no address outlives the context it came from (after cudaDeviceReset the
// module is loaded again and the array gets a new address).  The first call
// on a device loads the module there.
cudaError_t scratch_address(void **out) {
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" size_t swa_attn_decode_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

extern "C" swa_status swa_attn_decode_noalloc(swa_ctx *ctx, int32_t layer, int32_t bs,
                                              const int32_t *req_to_token, int64_t rt_stride,
                                              const int64_t *req_idx, const int64_t *seq_lens,
                                              int32_t max_seq_len, const void *plan,
                                              const void *q, const float *sinks, float sm_scale,
                                              float k_scale, float v_scale, void *out,
                                              swa_stream_t stream) {
  SWA_NVTX("swa_attn_decode_noalloc");
  if (!ctx) return SWA_ERR_INVALID;
  if (bs == 0) return SWA_OK;
  const size_t need = swa_attn_decode_ws_bytes(ctx, layer, bs, max_seq_len);
  if (need == 0) {
    swa::set_ctx_error(ctx, "swa_attn_decode_noalloc: invalid layer, batch or max_seq_len");
    return SWA_ERR_INVALID;
  }
  if (need > kNoAllocScratchBytes) {
    swa::set_ctx_error(ctx,
                       "swa_attn_decode_noalloc: this batch needs more split scratch than the "
                       "32 MiB fixed array holds; use swa_attn_decode with a workspace");
    return SWA_ERR_INVALID;
  }
  void *scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    swa::set_ctx_error(ctx, cudaGetErrorString(e));
    return SWA_ERR_CUDA;
  }
  const size_t zero = swa::decode_ws_zero_bytes(ctx, bs);
  e = cudaMemsetAsync(scratch, 0, zero < need ? zero : need, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    swa::set_ctx_error(ctx, cudaGetErrorString(e));
    return SWA_ERR_CUDA;
  }
  return swa_attn_decode(ctx, layer, bs, req_to_token, rt_stride, req_idx, seq_lens, max_seq_len,
                         plan, q, sinks, sm_scale, k_scale, v_scale, out, scratch,
                         kNoAllocScratchBytes, stream);
}
