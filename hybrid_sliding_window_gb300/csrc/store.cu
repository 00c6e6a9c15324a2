// KV store: scatter the new tokens' K/V rows into one layer's pool.
//
// Method: "SGLang source teardown (15)", section "who writes into the pages"
// (the write target carries the full and the SWA location, translated once
// per batch) and section "second mapping: the KV store" (FP8 is stored as
// bytes).  Rows land at the full slot on full layers and at the SWA slot on
// sliding / chunked layers; the envelope layout places slot t of pool-layer l
// at row kernel_id(t) + (2l | 2l+1) * ps ("SGLang PR #34602", implementation
// step 1).
//
// One thread moves 16 output bytes; consecutive threads cover consecutive
// bytes of a row, so both the read of k/v and the scattered row write are
// fully coalesced 16-byte accesses.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kv_codec.cuh"
#include "swa_internal.h"

namespace swa {
namespace {

struct StoreParams {
  const char *k;
  const char *v;
  int64_t n;
  const int64_t *full_loc;
  const int64_t *swa_loc;
  const int64_t *mapping;
  int64_t map_len;
  int in_full;
  int64_t pool_rows;      // pool_size + page_size
  KvAddr addr;
  int64_t chunks_per_row; // out row bytes / 16
  int dtype;
  float k_scale, v_scale;
  int32_t *err;
};

__global__ void k_store(StoreParams P) {
  const int64_t total = P.n * P.chunks_per_row * 2;
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t per_tok = P.chunks_per_row * 2;
    const int64_t i = g / per_tok;
    const int64_t rem = g % per_tok;
    const int is_v = rem >= P.chunks_per_row;
    const int64_t c = is_v ? rem - P.chunks_per_row : rem;
    int64_t slot;
    if (P.in_full) {
      slot = P.full_loc[i];
    } else if (P.swa_loc) {
      slot = P.swa_loc[i];
    } else {
      int64_t f = P.full_loc[i];
      if (f < 0) f += P.map_len;
      slot = (f >= 0 && f < P.map_len) ? P.mapping[f] : -1;
    }
    if (slot < 0 || slot >= P.pool_rows) {
      set_error(P.err, SWA_DEVERR_RANGE);
      continue;
    }
    char *dst = (is_v ? P.addr.v : P.addr.k) + kv_row(P.addr, slot) * P.addr.row_bytes + c * 16;
    const char *srcrow = is_v ? P.v : P.k;
    if (P.dtype == SWA_DTYPE_E4M3) {
      // 16 output bytes <- 16 bf16 inputs (32 bytes).
      const uint4 *src = reinterpret_cast<const uint4 *>(srcrow + (i * P.chunks_per_row + c) * 32);
      *reinterpret_cast<uint4 *>(dst) = e4m3_encode16(src[0], src[1], is_v ? P.v_scale : P.k_scale);
    } else {
      const uint4 *src = reinterpret_cast<const uint4 *>(srcrow + (i * P.chunks_per_row + c) * 16);
      *reinterpret_cast<uint4 *>(dst) = *src;
    }
  }
}

}  // namespace

cudaError_t launch_store(Ctx &c, int layer, const void *k, const void *v, int64_t n,
                         const int64_t *full_loc, const int64_t *swa_loc, float ks,
                         float vs, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const LayerInfo &L = c.layers[layer];
  StoreParams P;
  P.k = static_cast<const char *>(k);
  P.v = static_cast<const char *>(v);
  P.n = n;
  P.full_loc = full_loc;
  P.swa_loc = swa_loc;
  P.mapping = c.mapping;
  P.map_len = c.mapping_len;
  P.in_full = L.in_full ? 1 : 0;
  P.pool_rows = (L.in_full ? c.cfg.size_full : c.cfg.size_swa) + c.cfg.page_size;
  P.addr = L.addr;
  P.chunks_per_row = L.addr.row_bytes / 16;
  P.dtype = c.cfg.kv_dtype;
  P.k_scale = ks;
  P.v_scale = vs;
  P.err = c.err_word;
  int64_t total = n * P.chunks_per_row * 2;
  int64_t grid = (total + 255) / 256;
  int64_t cap = (int64_t)c.num_sms * 16;
  if (grid > cap) grid = cap;
  k_store<<<(int)grid, 256, 0, s>>>(P);
  return cudaGetLastError();
}

}  // namespace swa
