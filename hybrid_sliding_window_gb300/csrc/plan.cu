// Per-batch SWA page table, built once and read by every SWA-pool layer.
//
// Method: "SWA in SGLang" design note, section "attention backend: translate
// the index once before reading or writing": the backend turns the full-index
// page table into an SWA page table once per batch, and all SWA layers share
// it.  Here the table covers, per request, the positions an SWA-pool layer may
// read: lo = max(0, first query - Wx) .. hi = last query.  Since a page's
// positions share one SWA page (both pools allocate page-aligned runs), one
// mapping lookup per page suffices.
#include <cuda_runtime.h>

#include "swa_internal.h"

namespace swa {
namespace {

__global__ void k_plan(const int32_t *rt, int64_t rt_stride, const int64_t *req_idx,
                       const int64_t *pre, const int64_t *seq, int lookback, int ps,
                       const int64_t *mapping, int64_t map_len, int32_t *hdr,
                       int32_t *pages, int max_pages, int32_t *err) {
  const int b = blockIdx.x;
  const int64_t hi = seq[b] - 1;
  const int64_t first_q = pre ? pre[b] : hi;
  int64_t lo = first_q - lookback;
  if (lo < 0) lo = 0;
  if (hi < 0) {
    if (threadIdx.x == 0) {
      hdr[b * 4 + 0] = 0; hdr[b * 4 + 1] = -1; hdr[b * 4 + 2] = 0; hdr[b * 4 + 3] = 0;
    }
    return;
  }
  const int64_t first = lo / ps;
  int64_t n = hi / ps - first + 1;
  if (n > max_pages) {
    if (threadIdx.x == 0) set_error(err, SWA_DEVERR_RANGE);
    n = max_pages;
  }
  if (threadIdx.x == 0) {
    hdr[b * 4 + 0] = (int32_t)lo;
    hdr[b * 4 + 1] = (int32_t)hi;
    hdr[b * 4 + 2] = (int32_t)first;
    hdr[b * 4 + 3] = (int32_t)n;
  }
  const int64_t row = req_idx[b] * rt_stride;
  for (int64_t k = threadIdx.x; k < n; k += blockDim.x) {
    int64_t pos = (first + k) * ps;
    if (pos < lo) pos = lo;
    int64_t f = rt[row + pos];
    int64_t s = (f > 0 && f < map_len - 1) ? mapping[f] : 0;
    int32_t page = 0;
    if (s <= 0) set_error(err, SWA_DEVERR_WINDOW_EVICTED);
    else page = (int32_t)(s / ps);
    pages[(int64_t)b * max_pages + k] = page;
  }
}

}  // namespace

int plan_max_pages(const Ctx &c, int max_new) {
  const int ps = c.cfg.page_size;
  int64_t span = (int64_t)c.lookback + (max_new > 0 ? max_new : 1);
  return (int)((span + ps - 1) / ps + 1);
}

cudaError_t launch_plan(Ctx &c, int bs, const int32_t *rt, int64_t rt_stride,
                        const int64_t *req_idx, const int64_t *pre, const int64_t *seq,
                        int max_new, void *plan, cudaStream_t s) {
  if (bs == 0) return cudaSuccess;
  int maxp = plan_max_pages(c, max_new);
  int32_t *hdr = static_cast<int32_t *>(plan);
  int32_t *pages = hdr + (((int64_t)bs * 4 + 63) / 64) * 64;
  k_plan<<<bs, 128, 0, s>>>(rt, rt_stride, req_idx, pre, seq, c.lookback, c.cfg.page_size,
                            c.mapping, c.mapping_len, hdr, pages, maxp, c.err_word);
  return cudaGetLastError();
}

}  // namespace swa
