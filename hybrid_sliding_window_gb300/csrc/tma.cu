// TMA tensor maps over one layer's K and V rows, built once per context, and
// over an extend call's queries and outputs, built per call.
//
// A layer's K (or V) rows form a dense [rows][Hkv][D] array: the per-layer
// pool, or the layer's view of the page-major envelope (row = kernel-facing
// id).  One box is {128 bytes of one head's row, 1 head, min(ps, 64) rows}
// with the 128-byte swizzle, so a page (or 64 rows of one) lands in shared
// memory as [rows][128 B] blocks that ldmatrix and tcgen05 descriptors read
// without bank conflicts.
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include "swa_internal.h"

namespace swa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

void make_kv_tensor_maps(Ctx &c, int layer) {
  LayerInfo &L = c.layers[layer];
  L.tma = false;
  const int ps = c.cfg.page_size;
  if (c.cfg.kv_dtype == SWA_DTYPE_F32) return;
  if (ps < 16 || ps > 128 || (ps & (ps - 1))) return;
  const int esz = c.esize;
  const int row_bytes = c.cfg.head_dim * esz;       // one head's row
  if (row_bytes != 128 && row_bytes != 256) return;
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return;
  int64_t rows;
  if (L.addr.blocks == 0) {
    rows = (L.in_full ? c.cfg.size_full : c.cfg.size_swa) + ps;
  } else {
    rows = ((L.in_full ? c.cfg.size_full : c.cfg.size_swa) / ps + 1) * (int64_t)L.addr.blocks * ps;
  }
  cuuint64_t dims[3] = {(cuuint64_t)c.cfg.head_dim, (cuuint64_t)L.hkv, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)L.hkv * row_bytes};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esz), 1, (cuuint32_t)(ps < 64 ? ps : 64)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  for (int kv = 0; kv < 2; ++kv) {
    CUresult r = fn(kv ? &L.tmv : &L.tmk, dt, 3, kv ? (void *)L.addr.v : (void *)L.addr.k, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return;
  }
  L.tma = true;
}

bool make_qo_tensor_map(CUtensorMap *m, const void *x, int64_t nq, int hq, int d, int g) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || nq <= 0 || ((uintptr_t)x & 15) || g <= 0 || g > 128) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)nq};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(128 / g)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace swa
