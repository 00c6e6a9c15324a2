// Unified FULL/SWA pool allocated from both ends of one page range, with the
// per-side virtual-to-physical page tables the kernels translate through.
//
// Method: "SGLang source teardown (15)", allocator-family table
// (UnifiedSWATokenToKVPoolAllocator: FULL and SWA share one id space and are
// allocated from the two ends) and the note on UnifiedSWAAllocatorBase
// (shared virtual ids replace the full->SWA table; the allocation policy
// manages both sub-pools' budgets); SGLang PR #34602 summary,
// multi_ended_allocator.py (virtual_to_physical, translate_kv_loc_for_kernel
// with the tombstone clamped to the page-0 sink).
//
// Policy (this library's plain reading, where the pages stop): one physical
// page range 1..P; FULL takes pages upward from the low end (frontier `low`,
// the highest page it took), SWA downward from the high end (`high`, the
// lowest page it took); pages between the two frontiers belong to neither
// side.  A side reuses its released pages nearest its own end first (FULL the
// lowest, SWA the highest), then grows its frontier into the gap; after a
// release a frontier retracts over released pages that border it.  Virtual
// page ids (owned by the FULL side) come from a ring like the paged
// allocator's free list (front first; distinct released ids prepended in
// ascending order).
//
// GB300 design: released pages are a bitmap per side in the state blob, so a
// release is one atomicOr per page and a batch's reuse is one block-wide
// rank scan over the bitmap (the n lowest / highest set bits); every count
// that moves is a device counter; the host keeps a mirror of the counters
// that is exact after an allocation and is reloaded (one stream sync) on the
// first allocation after a release, because a retraction's length depends on
// which pages were released.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <new>
#include <string>

#include "swa_internal.h"

struct swa_unified {
  int64_t P = 0;
  int32_t ps = 1;
  int32_t max_batch = 1;
  int num_sms = 0;
  int64_t *ctr = nullptr;
  int64_t *v2p_f = nullptr, *v2p_s = nullptr, *vring = nullptr;
  uint32_t *bm_f = nullptr, *bm_s = nullptr;
  int64_t *ev_old = nullptr, *ev_new = nullptr, *ev_n = nullptr;
  int32_t *err = nullptr;
  // host mirror of the counters
  int64_t low = 0, high = 0, nrel_f = 0, nrel_s = 0, vcount = 0;
  bool stale = false;
  std::string msg;
};

namespace {

enum { C_LOW = SWA_UCTR_LOW, C_HIGH = SWA_UCTR_HIGH, C_RELF = SWA_UCTR_REL_FULL,
       C_RELS = SWA_UCTR_REL_SWA, C_VHEAD = SWA_UCTR_VHEAD, C_VCOUNT = SWA_UCTR_VCOUNT,
       C_ERR = SWA_UCTR_ERROR };

constexpr int64_t kMaxPages = 1700000;   // the release bitmap of the ids fits in shared memory

inline size_t al256(size_t x) { return (x + 255) / 256 * 256; }
__host__ __device__ inline int64_t words_of(int64_t P) { return (P + 1 + 31) / 32; }
__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Layout {
  size_t ctr, v2p_f, v2p_s, bm_f, bm_s, vring, ev, total;
};

Layout layout_of(int64_t P, int32_t max_batch) {
  Layout L;
  size_t off = 0;
  L.ctr = off; off = al256(off + 32 * sizeof(int64_t));
  L.v2p_f = off; off = al256(off + (size_t)(P + 1) * sizeof(int64_t));
  L.v2p_s = off; off = al256(off + (size_t)(P + 1) * sizeof(int64_t));
  L.bm_f = off; off = al256(off + (size_t)words_of(P) * 4);
  L.bm_s = off; off = al256(off + (size_t)words_of(P) * 4);
  L.vring = off; off = al256(off + (size_t)P * sizeof(int64_t));
  L.ev = off; off = al256(off + 3 * (size_t)max_batch * sizeof(int64_t));
  L.total = off;
  return L;
}

thread_local std::string g_create_msg;
swa_status fail(swa_unified *u, swa_status st, const std::string &m) {
  if (u) u->msg = m;
  else g_create_msg = m;
  return st;
}

#define U_TRY(u, expr)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(u, SWA_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(e_)); \
  } while (0)

// Exclusive block scan of one int64 per thread (blockDim.x a multiple of 32);
// returns the block total.
__device__ int64_t scan_excl(int64_t v, int64_t &excl) {
  __shared__ int64_t tot[32];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  int64_t x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (l >= o) x += y;
  }
  __syncthreads();
  if (l == 31) tot[w] = x;
  __syncthreads();
  if (w == 0) {
    int64_t t = l < nw ? tot[l] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (l >= o) t += y;
    }
    if (l < nw) tot[l] = t;
  }
  __syncthreads();
  excl = (w > 0 ? tot[w - 1] : 0) + x - v;
  const int64_t total = tot[nw - 1];
  __syncthreads();
  return total;
}

__device__ int64_t block_sum(int64_t v) {
  int64_t unused;
  return scan_excl(v, unused);
}

// Calls f(page, ascending rank) for every set bit of bm[0..words); each
// thread owns a contiguous run of words (f may clear bits of the word it is
// called for: only the owning thread reads it after the count).  Returns the
// number of set bits.
template <typename F>
__device__ int64_t for_ranked_bits(uint32_t *bm, int64_t words, F f) {
  const int64_t per = (words + blockDim.x - 1) / blockDim.x;
  const int64_t w0 = threadIdx.x * per, w1 = min(words, w0 + per);
  int64_t c = 0;
  for (int64_t w = w0; w < w1; ++w) c += __popc(bm[w]);
  int64_t r;
  const int64_t total = scan_excl(c, r);
  for (int64_t w = w0; w < w1; ++w) {
    uint32_t x = bm[w];
    while (x) {
      const int b = __ffs(x) - 1;
      x &= x - 1;
      f(w * 32 + b, r++);
    }
  }
  return total;
}

__global__ void k_u_init(int64_t P, int64_t *ctr, int64_t *v2p_f, int64_t *v2p_s, uint32_t *bm_f,
                         uint32_t *bm_s, int64_t *vring) {
  const int64_t words = words_of(P);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i <= P;
       i += (int64_t)gridDim.x * blockDim.x) {
    v2p_f[i] = i == 0 ? 0 : -1;
    v2p_s[i] = i == 0 ? 0 : -1;
    if (i < words) bm_f[i] = bm_s[i] = 0;
    if (i < P) vring[i] = i + 1;
  }
  if (blockIdx.x == 0 && threadIdx.x < 32) {
    int64_t v = 0;
    if (threadIdx.x == C_HIGH) v = P + 1;
    if (threadIdx.x == C_VCOUNT) v = P;
    ctr[threadIdx.x] = v;
  }
}

// Virtual slots of every request (one CTA per request): its output offset and
// first new virtual page are sums over the requests before it; positions in
// the open page continue after last_loc, the others fill the next virtual
// pages of the ring in request order.
__global__ void k_u_alloc_slots(int bs, const int64_t *pre, const int64_t *seq,
                                const int64_t *last_loc, int ps, int64_t P, const int64_t *ctr,
                                const int64_t *vring, int64_t *out, int32_t *rt,
                                int64_t rt_stride, const int64_t *req_idx, int32_t *err) {
  const int r = blockIdx.x;
  int64_t ext = 0, dp = 0;
  for (int i = threadIdx.x; i < r; i += blockDim.x) {
    ext += seq[i] - pre[i];
    dp += cdiv(seq[i], ps) - cdiv(pre[i], ps);
  }
  const int64_t out_off = block_sum(ext);
  const int64_t page_off = block_sum(dp);
  const int64_t p0 = pre[r], s0 = seq[r];
  const int64_t row = req_idx ? req_idx[r] * rt_stride : 0;
  int64_t last = -1;
  if (p0 > 0) last = last_loc ? last_loc[r] : (int64_t)rt[row + p0 - 1];
  const int64_t open_end = cdiv(p0, ps) * ps, first_new = cdiv(p0, ps);
  const int64_t head = ctr[C_VHEAD];
  for (int64_t t = p0 + threadIdx.x; t < s0; t += blockDim.x) {
    int64_t slot;
    if (t < open_end) {
      slot = last + 1 + (t - p0);
    } else {
      const int64_t k = page_off + (t / ps - first_new);
      slot = vring[(head + k) % P] * ps + t % ps;
    }
    out[out_off + (t - p0)] = slot;
    if (rt) {
      if (slot >= 0 && slot < ((int64_t)1 << 31)) rt[row + t] = (int32_t)slot;
      else swa::set_error(err, SWA_DEVERR_RANGE);
    }
  }
}

// Physical pages of the batch's new virtual pages (one CTA): the i-th new
// virtual page gets FULL's i-th lowest released page, else the page i - nF
// above the low frontier, and SWA's i-th highest released page, else the page
// i - nS below the high frontier; then the counters move.
__global__ void k_u_alloc_pages(int bs, const int64_t *pre, const int64_t *seq, int ps, int64_t P,
                                int64_t *ctr, int64_t *v2p_f, int64_t *v2p_s, uint32_t *bm_f,
                                uint32_t *bm_s, const int64_t *vring) {
  int64_t dp = 0;
  for (int i = threadIdx.x; i < bs; i += blockDim.x) dp += cdiv(seq[i], ps) - cdiv(pre[i], ps);
  const int64_t total = block_sum(dp);
  const int64_t head = ctr[C_VHEAD], low = ctr[C_LOW], high = ctr[C_HIGH];
  const int64_t relf = ctr[C_RELF], rels = ctr[C_RELS];
  const int64_t nF = min(total, relf), nS = min(total, rels);
  const int64_t words = words_of(P);
  __syncthreads();
  for_ranked_bits(bm_f, words, [&](int64_t page, int64_t rank) {
    if (rank < nF) {
      v2p_f[vring[(head + rank) % P]] = page;
      bm_f[page >> 5] &= ~(1u << (page & 31));
    }
  });
  for_ranked_bits(bm_s, words, [&](int64_t page, int64_t rank) {
    const int64_t d = rels - 1 - rank;           // rank from the high end
    if (d < nS) {
      v2p_s[vring[(head + d) % P]] = page;
      bm_s[page >> 5] &= ~(1u << (page & 31));
    }
  });
  for (int64_t i = threadIdx.x; i < total; i += blockDim.x) {
    const int64_t v = vring[(head + i) % P];
    if (i >= nF) v2p_f[v] = low + 1 + (i - nF);
    if (i >= nS) v2p_s[v] = high - 1 - (i - nS);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ctr[C_LOW] = low + (total - nF);
    ctr[C_HIGH] = high - (total - nS);
    ctr[C_RELF] = relf - nF;
    ctr[C_RELS] = rels - nS;
    ctr[C_VHEAD] = (head + total) % P;
    ctr[C_VCOUNT] -= total;
  }
}

// Release of the SWA page of the virtual page of each slot (a tombstone).
__device__ inline void release_swa_of(int64_t t, int ps, int64_t P, int64_t *v2p_s, uint32_t *bm_s,
                                      int64_t *ctr, int32_t *err) {
  const int64_t v = t >= 0 ? t / ps : -1;
  if (v < 1 || v > P) {
    swa::set_error(err, SWA_DEVERR_RANGE);
    return;
  }
  const int64_t p = v2p_s[v];
  if (p <= 0) return;
  const uint32_t bit = 1u << (p & 31);
  if (!(atomicOr(&bm_s[p >> 5], bit) & bit))
    atomicAdd(reinterpret_cast<unsigned long long *>(&ctr[C_RELS]), 1ull);
  v2p_s[v] = -1;
}

__global__ void k_u_free_swa(const int64_t *virt, int64_t n, int ps, int64_t P, int64_t *v2p_s,
                             uint32_t *bm_s, int64_t *ctr, int32_t *err) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    release_swa_of(virt[i], ps, P, v2p_s, bm_s, ctr, err);
}

// FULL pages and virtual ids of the slots' virtual pages (one CTA; runs after
// k_u_free_swa): each distinct live virtual page releases its FULL page into
// FULL's bitmap, and the distinct ids go back to the ring in ascending order
// just before its head.
__global__ void k_u_free_full(const int64_t *virt, int64_t n, int ps, int64_t P, int64_t *v2p_f,
                              uint32_t *bm_f, int64_t *vring, int64_t *ctr, int32_t *err) {
  extern __shared__ uint32_t vbm[];
  const int64_t words = words_of(P);
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) vbm[w] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t t = virt[i];
    const int64_t v = t >= 0 ? t / ps : -1;
    if (v < 1 || v > P) continue;          // flagged by k_u_free_swa
    const int64_t p = v2p_f[v];
    if (p <= 0) continue;
    const uint32_t bit = 1u << (p & 31);
    if (!(atomicOr(&bm_f[p >> 5], bit) & bit))
      atomicAdd(reinterpret_cast<unsigned long long *>(&ctr[C_RELF]), 1ull);
    atomicOr(&vbm[v >> 5], 1u << (v & 31));
    v2p_f[v] = -1;
  }
  __syncthreads();
  int64_t c = 0;
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) c += __popc(vbm[w]);
  const int64_t nv = block_sum(c);
  const int64_t head = ctr[C_VHEAD];
  for_ranked_bits(vbm, words, [&](int64_t v, int64_t rank) {
    vring[((head - nv + rank) % P + P) % P] = v;
  });
  __syncthreads();
  if (threadIdx.x == 0) {
    ctr[C_VHEAD] = ((head - nv) % P + P) % P;
    ctr[C_VCOUNT] += nv;
  }
}

// Frontier retraction (one thread): FULL's frontier moves down over released
// FULL pages that border it, SWA's moves up likewise; those pages leave the
// bitmaps and rejoin the gap.  Whole words are taken at a time.
__global__ void k_u_retract(int64_t P, int64_t *ctr, uint32_t *bm_f, uint32_t *bm_s, int do_full,
                            int do_swa) {
  if (threadIdx.x != 0) return;
  if (do_full) {
    int64_t low = ctr[C_LOW], taken = 0;
    while (low > 0) {
      const int64_t w = low >> 5;
      const int b = (int)(low & 31);
      const uint32_t below = b == 31 ? 0xffffffffu : ((1u << (b + 1)) - 1);   // bits 0..b
      const uint32_t x = bm_f[w] & below;
      // set bits from b downward: count leading ones of x shifted to the top
      const uint32_t top = x << (31 - b);
      const int run = __clz(~top);
      const int k = run > b + 1 ? b + 1 : run;
      if (k == 0) break;
      const uint32_t clr = (k == 32) ? 0xffffffffu : (((1u << k) - 1) << (b + 1 - k));
      bm_f[w] &= ~clr;
      low -= k;
      taken += k;
      if (k < b + 1) break;
    }
    ctr[C_LOW] = low;
    ctr[C_RELF] -= taken;
  }
  if (do_swa) {
    int64_t high = ctr[C_HIGH], taken = 0;
    while (high <= P) {
      const int64_t w = high >> 5;
      const int b = (int)(high & 31);
      const uint32_t x = bm_s[w] >> b;                   // bits b..31 moved to 0..
      const int avail = 32 - b;
      const int run = (~x) == 0 ? 32 : __ffs(~x) - 1;    // trailing ones
      int k = run > avail ? avail : run;
      if (high + k - 1 > P) k = (int)(P - high + 1);
      if (k == 0) break;
      const uint32_t clr = (k == 32) ? 0xffffffffu : (((1u << k) - 1) << b);
      bm_s[w] &= ~clr;
      high += k;
      taken += k;
      if (k < avail) break;
    }
    ctr[C_HIGH] = high;
    ctr[C_RELS] -= taken;
  }
}

// Eviction ranges (one thread per request), then one CTA per request
// releasing the SWA page of every page of its range.
__global__ void k_u_evict_plan(int bs, const int64_t *pre, const int64_t *evicted,
                               const int64_t *prot, int lookback, int ps, int interval, int radix,
                               int64_t *ev_old, int64_t *ev_new, int64_t *ev_n) {
  for (int b = threadIdx.x; b < bs; b += blockDim.x) {
    const int64_t ev = evicted[b];
    const int64_t bound = pre[b] - (radix ? (lookback > ps ? lookback : ps) : lookback);
    int64_t old_p = ev, new_p = ev, n = 0;
    if (!(interval > 0 && bound - ev < interval)) {
      new_p = bound > 0 ? (bound / ps) * ps : 0;
      const int64_t pr = prot ? prot[b] : 0;
      old_p = cdiv(ev > pr ? ev : pr, ps) * ps;
      if (new_p > old_p) n = (new_p - old_p) / ps;
    }
    ev_old[b] = old_p;
    ev_new[b] = n > 0 ? new_p : -1;
    ev_n[b] = n;
  }
}

__global__ void k_u_evict_apply(const int32_t *rt, int64_t rt_stride, const int64_t *req_idx,
                                int ps, int64_t P, const int64_t *ev_old, const int64_t *ev_n,
                                int64_t *v2p_s, uint32_t *bm_s, int64_t *ctr, int32_t *err) {
  const int b = blockIdx.x;
  const int64_t n = ev_n[b], old_p = ev_old[b], row = req_idx[b] * rt_stride;
  for (int64_t k = threadIdx.x; k < n; k += blockDim.x)
    release_swa_of(rt[row + old_p + k * ps], ps, P, v2p_s, bm_s, ctr, err);
}

__global__ void k_u_evict_commit(int bs, const int64_t *ev_new, const int64_t *ev_n,
                                 int64_t *evicted) {
  for (int b = threadIdx.x; b < bs; b += blockDim.x)
    if (ev_n[b] > 0) evicted[b] = ev_new[b];
}

// Host: reload the mirror from the device counters (synchronises the stream).
swa_status reload(swa_unified *u, cudaStream_t s) {
  int64_t h[8];
  U_TRY(u, cudaStreamSynchronize(s));
  U_TRY(u, cudaMemcpy(h, u->ctr, sizeof(h), cudaMemcpyDeviceToHost));
  u->low = h[C_LOW];
  u->high = h[C_HIGH];
  u->nrel_f = h[C_RELF];
  u->nrel_s = h[C_RELS];
  u->vcount = h[C_VCOUNT];
  u->stale = false;
  return SWA_OK;
}

bool fits(const swa_unified *u, int64_t n) {
  const int64_t gap = u->high - u->low - 1;
  return n <= u->vcount && std::max<int64_t>(0, n - u->nrel_f) +
                               std::max<int64_t>(0, n - u->nrel_s) <= gap;
}

int grid_for(int64_t n, int sms) {
  const int64_t g = std::min<int64_t>((n + 255) / 256, (int64_t)(sms > 0 ? sms : 148) * 8);
  return (int)std::max<int64_t>(1, g);
}

}  // namespace

extern "C" {

size_t swa_unified_state_bytes(int64_t num_pages, int32_t max_batch) {
  if (num_pages < 1 || max_batch < 1) return 0;
  return layout_of(num_pages, max_batch).total;
}

swa_status swa_unified_create(int64_t num_pages, int32_t page_size, int32_t max_batch,
                              void *state_dev, swa_stream_t stream, swa_unified **out) {
  SWA_NVTX("swa_unified_create");
  if (!out || !state_dev) return fail(nullptr, SWA_ERR_INVALID, "null state or output pointer");
  *out = nullptr;
  if (num_pages < 1 || page_size < 1 || max_batch < 1)
    return fail(nullptr, SWA_ERR_CONFIG, "num_pages, page_size and max_batch must be >= 1");
  if (num_pages > kMaxPages)
    return fail(nullptr, SWA_ERR_CONFIG, "more pages than the id release bitmap holds");
  if ((num_pages + 1) * page_size >= ((int64_t)1 << 31))
    return fail(nullptr, SWA_ERR_CONFIG, "virtual slots must fit req_to_token's int32");
  if (reinterpret_cast<uintptr_t>(state_dev) % 256)
    return fail(nullptr, SWA_ERR_INVALID, "state blob must be 256-byte aligned");
  swa_unified *u = new (std::nothrow) swa_unified();
  if (!u) return fail(nullptr, SWA_ERR_INVALID, "out of host memory");
  const Layout L = layout_of(num_pages, max_batch);
  char *base = static_cast<char *>(state_dev);
  u->P = num_pages;
  u->ps = page_size;
  u->max_batch = max_batch;
  u->ctr = reinterpret_cast<int64_t *>(base + L.ctr);
  u->v2p_f = reinterpret_cast<int64_t *>(base + L.v2p_f);
  u->v2p_s = reinterpret_cast<int64_t *>(base + L.v2p_s);
  u->bm_f = reinterpret_cast<uint32_t *>(base + L.bm_f);
  u->bm_s = reinterpret_cast<uint32_t *>(base + L.bm_s);
  u->vring = reinterpret_cast<int64_t *>(base + L.vring);
  int64_t *ev = reinterpret_cast<int64_t *>(base + L.ev);
  u->ev_old = ev;
  u->ev_new = ev + max_batch;
  u->ev_n = ev + 2 * (int64_t)max_batch;
  u->err = reinterpret_cast<int32_t *>(u->ctr + C_ERR);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&u->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) {
    k_u_init<<<grid_for(num_pages + 1, u->num_sms), 256, 0, (cudaStream_t)stream>>>(
        num_pages, u->ctr, u->v2p_f, u->v2p_s, u->bm_f, u->bm_s, u->vring);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    delete u;
    return fail(nullptr, SWA_ERR_CUDA, std::string("unified init: ") + cudaGetErrorString(e));
  }
  u->low = 0;
  u->high = num_pages + 1;
  u->vcount = num_pages;
  *out = u;
  return SWA_OK;
}

void swa_unified_destroy(swa_unified *u) { delete u; }

const char *swa_unified_last_error(const swa_unified *u) {
  return u ? u->msg.c_str() : g_create_msg.c_str();
}

swa_status swa_unified_state_pointers(const swa_unified *u, swa_unified_view *o) {
  if (!u || !o) return SWA_ERR_INVALID;
  o->v2p_full = u->v2p_f;
  o->v2p_swa = u->v2p_s;
  o->released_full = u->bm_f;
  o->released_swa = u->bm_s;
  o->virt_free = u->vring;
  o->counters = u->ctr;
  o->num_pages = u->P;
  return SWA_OK;
}

int64_t swa_unified_available_size(const swa_unified *u) {
  if (!u || u->stale) return -1;
  int64_t n = 0, lo = 0, hi = u->vcount;      // largest n that fits (fits is monotone)
  while (lo <= hi) {
    const int64_t mid = (lo + hi) / 2;
    if (fits(u, mid)) { n = mid; lo = mid + 1; } else { hi = mid - 1; }
  }
  return n * u->ps;
}

swa_status swa_unified_sync(swa_unified *u, swa_stream_t stream) {
  SWA_NVTX("swa_unified_sync");
  if (!u) return SWA_ERR_INVALID;
  return reload(u, (cudaStream_t)stream);
}

swa_status swa_unified_device_check(swa_unified *u, swa_stream_t stream, int32_t *err) {
  SWA_NVTX("swa_unified_device_check");
  if (!u) return SWA_ERR_INVALID;
  U_TRY(u, cudaStreamSynchronize((cudaStream_t)stream));
  int32_t w = 0;
  U_TRY(u, cudaMemcpy(&w, u->err, sizeof(w), cudaMemcpyDeviceToHost));
  U_TRY(u, cudaMemset(u->err, 0, sizeof(int32_t)));
  if (err) *err = w;
  if (w) return fail(u, SWA_ERR_DEVICE_CHECK, "device check flagged error bits " + std::to_string(w));
  return SWA_OK;
}

swa_status swa_unified_alloc_extend(swa_unified *u, int32_t bs, const int64_t *prefix_lens,
                                    const int64_t *seq_lens, const int64_t *last_loc,
                                    const int64_t *prefix_lens_host, const int64_t *seq_lens_host,
                                    int64_t *out_virt, int32_t *req_to_token, int64_t rt_stride,
                                    const int64_t *req_idx, swa_stream_t stream) {
  SWA_NVTX("swa_unified_alloc_extend");
  if (!u) return SWA_ERR_INVALID;
  if (bs < 0 || bs > u->max_batch) return fail(u, SWA_ERR_INVALID, "bs out of range");
  if (bs == 0) return SWA_OK;
  if (!prefix_lens || !seq_lens || !prefix_lens_host || !seq_lens_host)
    return fail(u, SWA_ERR_INVALID, "null lengths");
  if (!last_loc && !req_to_token) return fail(u, SWA_ERR_INVALID, "need last_loc or req_to_token");
  if (req_to_token && (!req_idx || rt_stride < 1))
    return fail(u, SWA_ERR_INVALID, "req_to_token needs req_idx");
  const int64_t ps = u->ps;
  int64_t total = 0, n_tok = 0;
  for (int b = 0; b < bs; ++b) {
    const int64_t pr = prefix_lens_host[b], sq = seq_lens_host[b];
    if (pr < 0 || sq < pr) return fail(u, SWA_ERR_INVALID, "need 0 <= prefix <= seq");
    if (req_to_token && sq > rt_stride) return fail(u, SWA_ERR_INVALID, "seq exceeds req_to_token row");
    total += cdiv(sq, ps) - cdiv(pr, ps);
    n_tok += sq - pr;
  }
  if (n_tok == 0) return SWA_OK;
  if (!out_virt) return fail(u, SWA_ERR_INVALID, "null output");
  cudaStream_t s = (cudaStream_t)stream;
  if (u->stale) {
    const swa_status st = reload(u, s);
    if (st != SWA_OK) return st;
  }
  if (!fits(u, total)) return fail(u, SWA_ERR_NOMEM, "not enough pages between the two ends");
  k_u_alloc_slots<<<bs, 256, 0, s>>>(bs, prefix_lens, seq_lens, last_loc, u->ps, u->P, u->ctr,
                                     u->vring, out_virt, req_to_token, rt_stride, req_idx, u->err);
  U_TRY(u, cudaGetLastError());
  if (total > 0) {
    k_u_alloc_pages<<<1, 1024, 0, s>>>(bs, prefix_lens, seq_lens, u->ps, u->P, u->ctr, u->v2p_f,
                                       u->v2p_s, u->bm_f, u->bm_s, u->vring);
    U_TRY(u, cudaGetLastError());
  }
  const int64_t nf = std::min(total, u->nrel_f), ns = std::min(total, u->nrel_s);
  u->low += total - nf;
  u->high -= total - ns;
  u->nrel_f -= nf;
  u->nrel_s -= ns;
  u->vcount -= total;
  return SWA_OK;
}

swa_status swa_unified_free_swa(swa_unified *u, const int64_t *virt, int64_t n,
                                swa_stream_t stream) {
  SWA_NVTX("swa_unified_free_swa");
  if (!u || n < 0 || (n > 0 && !virt)) return fail(u, SWA_ERR_INVALID, "bad free_swa args");
  if (n == 0) return SWA_OK;
  cudaStream_t s = (cudaStream_t)stream;
  k_u_free_swa<<<grid_for(n, u->num_sms), 256, 0, s>>>(virt, n, u->ps, u->P, u->v2p_s, u->bm_s,
                                                      u->ctr, u->err);
  k_u_retract<<<1, 32, 0, s>>>(u->P, u->ctr, u->bm_f, u->bm_s, 0, 1);
  U_TRY(u, cudaGetLastError());
  u->stale = true;
  return SWA_OK;
}

swa_status swa_unified_free(swa_unified *u, const int64_t *virt, int64_t n, swa_stream_t stream) {
  SWA_NVTX("swa_unified_free");
  if (!u || n < 0 || (n > 0 && !virt)) return fail(u, SWA_ERR_INVALID, "bad free args");
  if (n == 0) return SWA_OK;
  cudaStream_t s = (cudaStream_t)stream;
  k_u_free_swa<<<grid_for(n, u->num_sms), 256, 0, s>>>(virt, n, u->ps, u->P, u->v2p_s, u->bm_s,
                                                      u->ctr, u->err);
  const size_t smem = (size_t)words_of(u->P) * 4;
  U_TRY(u, cudaFuncSetAttribute(k_u_free_full, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem));
  k_u_free_full<<<1, 1024, smem, s>>>(virt, n, u->ps, u->P, u->v2p_f, u->bm_f, u->vring, u->ctr,
                                      u->err);
  k_u_retract<<<1, 32, 0, s>>>(u->P, u->ctr, u->bm_f, u->bm_s, 1, 1);
  U_TRY(u, cudaGetLastError());
  u->stale = true;
  return SWA_OK;
}

swa_status swa_unified_evict_swa(swa_unified *u, int32_t bs, int32_t window_excl,
                                 const int32_t *req_to_token, int64_t rt_stride,
                                 const int64_t *req_idx, const int64_t *pre_lens,
                                 int64_t *evicted, const int64_t *protected_lens,
                                 const int64_t *pre_lens_host, int64_t *evicted_host,
                                 const int64_t *protected_host, int32_t interval, int32_t radix,
                                 swa_stream_t stream) {
  SWA_NVTX("swa_unified_evict_swa");
  if (!u) return SWA_ERR_INVALID;
  if (bs < 0 || bs > u->max_batch) return fail(u, SWA_ERR_INVALID, "bs out of range");
  if (bs == 0) return SWA_OK;
  if (!req_to_token || !req_idx || !pre_lens || !evicted || !pre_lens_host || !evicted_host ||
      interval < 0 || window_excl < 0)
    return fail(u, SWA_ERR_INVALID, "bad evict args");
  const int64_t ps = u->ps;
  const int64_t lb = radix ? std::max<int64_t>(window_excl, ps) : window_excl;
  int64_t total = 0;
  std::string err;
  for (int b = 0; b < bs; ++b) {
    const int64_t ev = evicted_host[b], bound = pre_lens_host[b] - lb;
    if (interval > 0 && bound - ev < interval) continue;
    const int64_t nw = bound > 0 ? bound / ps * ps : 0;
    const int64_t prot = protected_host ? protected_host[b] : 0;
    const int64_t old = cdiv(std::max(ev, prot), ps) * ps;
    if (nw > old) {
      if (nw > rt_stride) return fail(u, SWA_ERR_INVALID, "eviction range beyond req_to_token row");
      total += (nw - old) / ps;
    }
  }
  if (total == 0) return SWA_OK;
  cudaStream_t s = (cudaStream_t)stream;
  k_u_evict_plan<<<1, 256, 0, s>>>(bs, pre_lens, evicted, protected_lens, window_excl, u->ps,
                                   interval, radix, u->ev_old, u->ev_new, u->ev_n);
  k_u_evict_apply<<<bs, 256, 0, s>>>(req_to_token, rt_stride, req_idx, u->ps, u->P, u->ev_old,
                                     u->ev_n, u->v2p_s, u->bm_s, u->ctr, u->err);
  k_u_retract<<<1, 32, 0, s>>>(u->P, u->ctr, u->bm_f, u->bm_s, 0, 1);
  k_u_evict_commit<<<1, 256, 0, s>>>(bs, u->ev_new, u->ev_n, evicted);
  U_TRY(u, cudaGetLastError());
  for (int b = 0; b < bs; ++b) {
    const int64_t ev = evicted_host[b], bound = pre_lens_host[b] - lb;
    if (interval > 0 && bound - ev < interval) continue;
    const int64_t nw = bound > 0 ? bound / ps * ps : 0;
    const int64_t prot = protected_host ? protected_host[b] : 0;
    if (nw > cdiv(std::max(ev, prot), ps) * ps) evicted_host[b] = nw;
  }
  u->stale = true;
  return SWA_OK;
}

}  // extern "C"
