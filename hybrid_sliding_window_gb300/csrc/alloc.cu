// Two-pool page allocator, full->SWA mapping, release and eviction kernels.
//
// Method: "SWA in SGLang" design note, sections "two pools and the mapping"
// and "runtime: returning slid-out KV"; "SGLang source teardown (15)",
// sections "alloc_extend", "alloc_decode", "free, dedupe and free_group",
// "_release_page_ids".
//
// GB300 design: each free list is a device ring of page ids whose front is
// `head`; allocation advances head, a release writes the freed ids in
// ascending order just before head (the pages' "prepend"), so nothing is
// ever copied or re-allocated.  Dedupe + ascending order come from a bitmap
// over page ids in shared memory (a set bit per page, then a block-wide
// compaction), which replaces a device sort.  All counts that decide a
// launch are known on the host; all positions are computed on the device
// from device arrays, so the kernels can be replayed from a CUDA graph.
#include <cuda_runtime.h>
#include <stdint.h>

#include "swa_internal.h"

namespace swa {
namespace {

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
__device__ inline int64_t ring_pos(int64_t head, int64_t i, int64_t cap) {
  int64_t x = (head + i) % cap;
  return x < 0 ? x + cap : x;
}

// Block-wide sum of two int64 values (blockDim.x multiple of 32, <= 1024).
__device__ inline void block_sum2(int64_t &a, int64_t &b) {
  __shared__ int64_t sa[32], sb[32];
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_down_sync(0xffffffffu, a, o);
    b += __shfl_down_sync(0xffffffffu, b, o);
  }
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) { sa[w] = a; sb[w] = b; }
  __syncthreads();
  int nw = blockDim.x >> 5;
  if (w == 0) {
    a = l < nw ? sa[l] : 0;
    b = l < nw ? sb[l] : 0;
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_down_sync(0xffffffffu, a, o);
      b += __shfl_down_sync(0xffffffffu, b, o);
    }
    if (l == 0) { sa[0] = a; sb[0] = b; }
  }
  __syncthreads();
  a = sa[0];
  b = sb[0];
  __syncthreads();
}

// Exclusive block scan of one int64 per thread; returns the block total.
__device__ inline int64_t block_excl_scan(int64_t v, int64_t &excl) {
  __shared__ int64_t warp_tot[32];
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  int64_t x = v;
  for (int o = 1; o < 32; o <<= 1) {
    int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (l >= o) x += y;
  }
  __syncthreads();
  if (l == 31) warp_tot[w] = x;
  __syncthreads();
  int nw = blockDim.x >> 5;
  if (w == 0) {
    int64_t t = l < nw ? warp_tot[l] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (l >= o) t += y;
    }
    if (l < nw) warp_tot[l] = t;  // inclusive prefix of warp totals
  }
  __syncthreads();
  int64_t before = w > 0 ? warp_tot[w - 1] : 0;
  excl = before + x - v;
  int64_t total = warp_tot[nw - 1];
  __syncthreads();
  return total;
}

// ------------------------------------------------------------------ init ---
__global__ void k_init_state(int64_t *mapping, int64_t map_len, PoolDev full,
                             PoolDev swa, const int64_t *init_full,
                             const int64_t *init_swa, int64_t *counters) {
  int64_t n = map_len;
  if (full.cap > n) n = full.cap;
  if (swa.cap > n) n = swa.cap;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < map_len) mapping[i] = (i == map_len - 1) ? -1 : 0;
    if (i < full.cap) full.ring[i] = init_full ? init_full[i] : i + 1;
    if (i < swa.cap) swa.ring[i] = init_swa ? init_swa[i] : i + 1;
  }
  if (blockIdx.x == 0 && threadIdx.x < 64) {
    int64_t v = 0;
    if (threadIdx.x == SWA_CTR_FULL_COUNT) v = full.cap;
    if (threadIdx.x == SWA_CTR_SWA_COUNT) v = swa.cap;
    counters[threadIdx.x] = v;
  }
}

// ------------------------------------------------------------ alloc_extend ---
// One CTA per request.  Request r's output offset and first new page are the
// sums of the extend lengths / new-page counts of requests 0..r-1; its slots
// follow last_loc inside the open page, then fill pages taken from the free
// ring in request order (slot = page * ps + t % ps).
__global__ void k_alloc_extend(int bs, const int64_t *pre, const int64_t *seq,
                               const int64_t *last_loc, int ps, PoolDev full,
                               PoolDev swa, int64_t *mapping, int64_t map_len,
                               int64_t *out_full, int64_t *out_swa, int32_t *rt,
                               int64_t rt_stride, const int64_t *req_idx,
                               int32_t *err) {
  const int r = blockIdx.x;
  int64_t ext = 0, dp = 0;
  for (int i = threadIdx.x; i < r; i += blockDim.x) {
    int64_t s = seq[i];
    int64_t p = pre ? pre[i] : s - 1;
    ext += s - p;
    dp += cdiv(s, ps) - cdiv(p, ps);
  }
  block_sum2(ext, dp);
  const int64_t out_off = ext, page_off = dp;
  const int64_t s_r = seq[r];
  const int64_t p_r = pre ? pre[r] : s_r - 1;
  int64_t last_f;
  if (last_loc) {
    last_f = last_loc[r];
  } else {
    last_f = p_r > 0 ? (int64_t)rt[req_idx[r] * rt_stride + p_r - 1] : -1;
  }
  int64_t last_s;
  if (last_f == -1) {
    last_s = mapping[map_len - 1];  // the trailing -1 sentinel
  } else if (last_f < 0 || last_f >= map_len - 1) {
    last_s = -1;
    if (threadIdx.x == 0) set_error(err, SWA_DEVERR_RANGE);
  } else {
    last_s = mapping[last_f];
  }
  const int64_t open_end = cdiv(p_r, ps) * ps;
  // Per-request ring: the SWA slot is a function of (request slot, position).
  const bool ring = swa.ring_cost > 0;
  int64_t ring_base = -1;
  if (ring) {
    const int64_t rq = req_idx[r];
    if (rq >= 0 && rq < swa.ring_slots) ring_base = ps + rq * swa.ring_cost;
    else if (threadIdx.x == 0) set_error(err, SWA_DEVERR_RANGE);
  }
  if (threadIdx.x == 0 && p_r < open_end && (last_f < 0 || (!ring && last_s <= 0)))
    set_error(err, SWA_DEVERR_RANGE);
  const int64_t first_new = cdiv(p_r, ps);
  const int64_t hf = *full.head, hs = *swa.head;
  const int64_t row = rt ? req_idx[r] * rt_stride : 0;
  for (int64_t t = p_r + threadIdx.x; t < s_r; t += blockDim.x) {
    int64_t f, s;
    if (t < open_end) {
      f = last_f + 1 + (t - p_r);
      s = last_s + 1 + (t - p_r);
    } else {
      int64_t k = t / ps - first_new;
      int64_t pf = full.ring[ring_pos(hf, page_off + k, full.cap)];
      f = pf * ps + t % ps;
      s = ring ? 0 : swa.ring[ring_pos(hs, page_off + k, swa.cap)] * ps + t % ps;
    }
    if (ring) s = ring_base >= 0 ? ring_base + t % swa.ring_cost : 0;
    int64_t o = out_off + (t - p_r);
    out_full[o] = f;
    if (out_swa) out_swa[o] = s;
    if (f > 0 && f < map_len - 1) {
      mapping[f] = s;
    } else {
      set_error(err, SWA_DEVERR_RANGE);
    }
    if (rt) rt[row + t] = (int32_t)f;
  }
}

// Advance both rings by the total number of new pages of the batch.
__global__ void k_alloc_commit(int bs, const int64_t *pre, const int64_t *seq,
                               int ps, PoolDev full, PoolDev swa) {
  int64_t dp = 0, unused = 0;
  for (int i = threadIdx.x; i < bs; i += blockDim.x) {
    int64_t s = seq[i];
    int64_t p = pre ? pre[i] : s - 1;
    dp += cdiv(s, ps) - cdiv(p, ps);
  }
  block_sum2(dp, unused);
  if (threadIdx.x == 0) {
    *full.head = (*full.head + dp) % full.cap;
    *full.count -= dp;
    if (swa.ring_cost == 0) {   // per-request rings take no pages
      *swa.head = (*swa.head + dp) % swa.cap;
      *swa.count -= dp;
    }
  }
}

// Plain alloc(need): whole pages, same count from both rings.
__global__ void k_alloc_pages(int64_t need, int ps, PoolDev full, PoolDev swa,
                              int64_t *mapping, int64_t map_len,
                              int64_t *out_full, int64_t *out_swa, int32_t *err) {
  const int64_t hf = *full.head, hs = *swa.head;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < need;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t f = full.ring[ring_pos(hf, i / ps, full.cap)] * ps + i % ps;
    int64_t s = swa.ring[ring_pos(hs, i / ps, swa.cap)] * ps + i % ps;
    out_full[i] = f;
    if (out_swa) out_swa[i] = s;
    if (f > 0 && f < map_len - 1) mapping[f] = s;
    else set_error(err, SWA_DEVERR_RANGE);
  }
}

__global__ void k_advance(PoolDev full, PoolDev swa, int64_t n) {
  *full.head = (*full.head + n) % full.cap;
  *full.count -= n;
  *swa.head = (*swa.head + n) % swa.cap;
  *swa.count -= n;
}

// ----------------------------------------------------- bitmap compaction ---
// Writes the set bits of bm[0..words) in ascending order (page id = bit index)
// to dst(j) for j = 0..total-1 and returns total (all threads).  Each thread
// owns a contiguous word range.
template <typename Dst>
__device__ int64_t compact_bitmap(const uint32_t *bm, int64_t words, Dst dst) {
  const int64_t per = (words + blockDim.x - 1) / blockDim.x;
  const int64_t w0 = threadIdx.x * per;
  const int64_t w1 = min(words, w0 + per);
  int64_t c = 0;
  for (int64_t w = w0; w < w1; ++w) c += __popc(bm[w]);
  int64_t off;
  int64_t total = block_excl_scan(c, off);
  for (int64_t w = w0; w < w1; ++w) {
    uint32_t x = bm[w];
    while (x) {
      int b = __ffs(x) - 1;
      x &= x - 1;
      dst(off++, w * 32 + b);
    }
  }
  return total;
}

// need_sort merge: free := sort(free U staged).
__global__ void k_merge_sorted(PoolDev pool) {
  extern __shared__ uint32_t bm[];
  const int64_t words = (pool.cap + 1 + 31) / 32;
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) bm[w] = 0;
  __syncthreads();
  const int64_t head = *pool.head, count = *pool.count, ns = *pool.nstaged;
  for (int64_t i = threadIdx.x; i < count; i += blockDim.x) {
    int64_t p = pool.ring[ring_pos(head, i, pool.cap)];
    atomicOr(&bm[p >> 5], 1u << (p & 31));
  }
  for (int64_t i = threadIdx.x; i < ns; i += blockDim.x) {
    int64_t p = pool.staged[i];
    atomicOr(&bm[p >> 5], 1u << (p & 31));
  }
  __syncthreads();
  int64_t *ring = pool.ring;
  int64_t total = compact_bitmap(bm, words, [&](int64_t j, int64_t page) { ring[j] = page; });
  __syncthreads();
  if (threadIdx.x == 0) {
    *pool.head = 0;
    *pool.count = total;
    *pool.nstaged = 0;
  }
}

// Release the distinct pages of a set (bits already in bm) into `pool`:
// ascending ids either staged (need_sort) or written just before head.
__device__ void release_bitmap(const uint32_t *bm, PoolDev pool, bool need_sort,
                               int64_t expect, int32_t *err) {
  const int64_t words = (pool.cap + 1 + 31) / 32;
  // Count first, so the ring position of the first page is known.
  int64_t c = 0;
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) c += __popc(bm[w]);
  int64_t unused;
  const int64_t n_u = block_excl_scan(c, unused);
  const int64_t head = *pool.head;
  const int64_t ns = *pool.nstaged;
  __syncthreads();
  if (need_sort) {
    int64_t *st = pool.staged;
    compact_bitmap(bm, words, [&](int64_t j, int64_t page) { st[ns + j] = page; });
  } else {
    int64_t *ring = pool.ring;
    const int64_t cap = pool.cap;
    compact_bitmap(bm, words, [&](int64_t j, int64_t page) {
      ring[ring_pos(head, j - n_u, cap)] = page;
    });
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (need_sort) {
      *pool.nstaged = ns + n_u;
    } else {
      *pool.head = ((head - n_u) % pool.cap + pool.cap) % pool.cap;
      *pool.count += n_u;
    }
    if (expect >= 0 && expect != n_u) set_error(err, SWA_DEVERR_COUNT);
  }
  __syncthreads();
}

// free(idx) [do_full] then free_swa(idx): single CTA, bitmap in shared memory.
__global__ void k_release(const int64_t *idx, int64_t n, int do_full, int ps,
                          PoolDev full, PoolDev swa, int64_t *mapping,
                          int64_t map_len, int need_sort, int64_t expect_full,
                          int64_t expect_swa, int32_t *err) {
  extern __shared__ uint32_t bm[];
  if (do_full) {
    const int64_t words = (full.cap + 1 + 31) / 32;
    for (int64_t w = threadIdx.x; w < words; w += blockDim.x) bm[w] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      int64_t page = idx[i] / ps;
      if (idx[i] < 0 || page < 1 || page > full.cap) {
        set_error(err, SWA_DEVERR_RANGE);
        continue;
      }
      atomicOr(&bm[page >> 5], 1u << (page & 31));
    }
    __syncthreads();
    release_bitmap(bm, full, need_sort, expect_full, err);
  }
  if (swa.ring_cost > 0) {   // per-request rings: nothing to release, only unmap
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      int64_t f = idx[i];
      if (f >= 0 && f < map_len - 1) mapping[f] = 0;
      else set_error(err, SWA_DEVERR_RANGE);
    }
    return;
  }
  const int64_t words = (swa.cap + 1 + 31) / 32;
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) bm[w] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    int64_t f = idx[i];
    if (f < 0 || f >= map_len - 1) {
      set_error(err, SWA_DEVERR_RANGE);
      continue;
    }
    int64_t s = mapping[f];
    if (s > 0) {
      int64_t page = s / ps;
      if (page <= swa.cap) atomicOr(&bm[page >> 5], 1u << (page & 31));
      else set_error(err, SWA_DEVERR_RANGE);
    }
  }
  __syncthreads();
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    int64_t f = idx[i];
    if (f >= 0 && f < map_len - 1) mapping[f] = 0;
  }
  __syncthreads();
  release_bitmap(bm, swa, need_sort, expect_swa, err);
}

// -------------------------------------------------------------- eviction ---
// SWA page of request position t, or 0 when its mapping is not live (never
// allocated, or already released by free_swa).
__device__ inline int64_t live_swa_page(const int32_t *rt, int64_t row, int64_t t,
                                        const int64_t *mapping, int64_t map_len, int ps) {
  const int64_t f = rt[row + t];
  const int64_t s = (f > 0 && f < map_len - 1) ? mapping[f] : 0;
  return s > 0 ? s / ps : 0;
}

// Pass 1 (one CTA per request): the page-aligned range [old, new) and, for a
// paged SWA pool, how many of its pages still hold a live SWA page (one
// representative position per page: the range is page aligned and the ps
// positions of one request page share one SWA page).  free_swa skips
// positions whose mapping is not live, so only live pages are released; a
// range with dead pages disagrees with the host's count (SWA_DEVERR_COUNT).
__global__ void k_evict_plan(int bs, const int32_t *rt, int64_t rt_stride,
                             const int64_t *req_idx, const int64_t *pre,
                             const int64_t *evicted, const int64_t *prot, int lookback, int ps,
                             int interval, int radix, const int64_t *mapping, int64_t map_len,
                             bool count_live, EvictScratch sc, int32_t *err) {
  __shared__ int64_t s_old, s_n;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    const int64_t ev = evicted[b];
    const int64_t bound = pre[b] - (radix ? (lookback > ps ? lookback : ps) : lookback);
    int64_t old_p = ev, new_p = ev, n = 0;
    if (!(interval > 0 && bound - ev < interval)) {
      new_p = bound > 0 ? (bound / ps) * ps : 0;
      const int64_t pr = prot ? prot[b] : 0;
      old_p = cdiv(ev > pr ? ev : pr, ps) * ps;
      if (new_p > old_p) n = (new_p - old_p) / ps;
    }
    sc.old_pos[b] = old_p;
    sc.new_pos[b] = n > 0 ? new_p : -1;
    sc.npages[b] = n;
    s_old = old_p;
    s_n = count_live ? n : 0;
  }
  __syncthreads();
  const int64_t n = s_n, old_p = s_old, row = req_idx[b] * rt_stride;
  int64_t live = 0, unused = 0;
  for (int64_t k = threadIdx.x; k < n; k += blockDim.x)
    live += live_swa_page(rt, row, old_p + k * ps, mapping, map_len, ps) > 0;
  block_sum2(live, unused);
  if (threadIdx.x == 0) {
    sc.nlive[b] = live;
    if (live != n) set_error(err, SWA_DEVERR_COUNT);
  }
}

// Pass 2 (one CTA per request): the live SWA pages of the range, ascending
// (set bits of a bitmap over the pool's page ids in shared memory, then a
// block-wide compaction), written at the request's place in the freed run -
// later requests ahead of earlier ones without need_sort (sequential
// prepends), in batch order into the staging list with need_sort - and the
// range's mapping entries zeroed.
__global__ void k_evict_apply(int bs, const int32_t *rt, int64_t rt_stride,
                              const int64_t *req_idx, int ps, PoolDev swa,
                              int64_t *mapping, int64_t map_len, EvictScratch sc,
                              int need_sort, int32_t *err) {
  extern __shared__ uint32_t bm[];
  const int b = blockIdx.x;
  const int64_t n = sc.npages[b];
  if (n == 0) return;
  const int64_t old_p = sc.old_pos[b], new_p = sc.new_pos[b];
  const int64_t row = req_idx[b] * rt_stride;
  if (swa.ring_cost > 0) {   // per-request rings: the slid-out tokens are only unmapped
    for (int64_t t = old_p + threadIdx.x; t < new_p; t += blockDim.x) {
      int64_t f = rt[row + t];
      if (f > 0 && f < map_len - 1) mapping[f] = 0;
    }
    return;
  }
  // This request's offset in the batch's freed run, and the run's length.
  int64_t before = 0, total = 0;
  for (int i = threadIdx.x; i < bs; i += blockDim.x) {
    const int64_t v = sc.nlive[i];
    total += v;
    if (need_sort ? i < b : i > b) before += v;
  }
  block_sum2(before, total);
  const int64_t words = (swa.cap + 1 + 31) / 32;
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) bm[w] = 0;
  __syncthreads();
  for (int64_t k = threadIdx.x; k < n; k += blockDim.x) {
    const int64_t page = live_swa_page(rt, row, old_p + k * ps, mapping, map_len, ps);
    if (page > swa.cap) set_error(err, SWA_DEVERR_RANGE);
    else if (page > 0) atomicOr(&bm[page >> 5], 1u << (page & 31));
  }
  __syncthreads();
  if (need_sort) {
    int64_t *st = swa.staged + *swa.nstaged + before;
    compact_bitmap(bm, words, [&](int64_t j, int64_t page) { st[j] = page; });
  } else {
    const int64_t head = *swa.head, cap = swa.cap;
    int64_t *ring = swa.ring;
    compact_bitmap(bm, words, [&](int64_t j, int64_t page) {
      ring[ring_pos(head, before + j - total, cap)] = page;
    });
  }
  __syncthreads();   // every mapping read above precedes the zeroing below
  for (int64_t t = old_p + threadIdx.x; t < new_p; t += blockDim.x) {
    int64_t f = rt[row + t];
    if (f > 0 && f < map_len - 1) mapping[f] = 0;
  }
}

// Pass 3 (one CTA): move head / staged count, record the new evicted lengths.
__global__ void k_evict_commit(int bs, int64_t *evicted, PoolDev swa,
                               EvictScratch sc, int need_sort) {
  int64_t total = 0, unused = 0;
  for (int b = threadIdx.x; b < bs; b += blockDim.x) {
    if (sc.npages[b] > 0) evicted[b] = sc.new_pos[b];
    total += sc.nlive[b];
  }
  block_sum2(total, unused);
  if (threadIdx.x == 0 && swa.ring_cost == 0) {
    if (need_sort) {
      *swa.nstaged += total;
    } else {
      *swa.head = ((*swa.head - total) % swa.cap + swa.cap) % swa.cap;
      *swa.count += total;
    }
  }
}

// ------------------------------------------- translate for the kernels ---
// Virtual token id -> kernel-facing row id through a virtual-to-physical page
// table: phys * (ps * multiplier) + t % ps, a tombstone page (-1) clamped to 0.
__global__ void k_translate_for_kernel(const int64_t *v2p, int64_t n_pages, const int64_t *virt,
                                       int64_t n, int64_t ps, int64_t stride, int64_t *out,
                                       int32_t *err) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = virt[i];
    const int64_t page = t >= 0 ? t / ps : -1;
    if (page < 0 || page >= n_pages) {
      if (err) atomicOr(err, SWA_DEVERR_RANGE);
      out[i] = 0;
      continue;
    }
    const int64_t id = v2p[page] * stride + t % ps;
    out[i] = id > 0 ? id : 0;
  }
}

// ------------------------------------------------------------- translate ---
__global__ void k_translate(const int64_t *full_loc, int64_t n, const int64_t *mapping,
                            int64_t map_len, int64_t *swa_loc, int32_t *err) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t f = full_loc[i];
    if (f < 0) f += map_len;  // -1 reads the sentinel
    if (f < 0 || f >= map_len) {
      set_error(err, SWA_DEVERR_RANGE);
      swa_loc[i] = 0;
    } else {
      swa_loc[i] = mapping[f];
    }
  }
}

inline int grid_for(int64_t n, int block, int sms) {
  int64_t g = (n + block - 1) / block;
  int64_t cap = (int64_t)sms * 8;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_init_state(Ctx &c, const int64_t *init_full, const int64_t *init_swa,
                              cudaStream_t s) {
  int64_t n = c.mapping_len;
  if (c.np_full > n) n = c.np_full;
  if (c.np_swa > n) n = c.np_swa;
  k_init_state<<<grid_for(n, 256, c.num_sms), 256, 0, s>>>(
      c.mapping, c.mapping_len, c.full, c.swa, init_full, init_swa, c.counters);
  return cudaGetLastError();
}

cudaError_t launch_alloc_extend(Ctx &c, int bs, const int64_t *pre, const int64_t *seq,
                                const int64_t *last_loc, int64_t *out_full,
                                int64_t *out_swa, int32_t *rt, int64_t rt_stride,
                                const int64_t *req_idx, int max_new, cudaStream_t s) {
  (void)max_new;
  if (bs == 0) return cudaSuccess;
  k_alloc_extend<<<bs, 256, 0, s>>>(bs, pre, seq, last_loc, c.cfg.page_size, c.full, c.swa,
                                     c.mapping, c.mapping_len, out_full, out_swa, rt,
                                     rt_stride, req_idx, c.err_word);
  k_alloc_commit<<<1, 256, 0, s>>>(bs, pre, seq, c.cfg.page_size, c.full, c.swa);
  return cudaGetLastError();
}

cudaError_t launch_alloc_pages(Ctx &c, int64_t need, int64_t *out_full, int64_t *out_swa,
                               cudaStream_t s) {
  if (need == 0) return cudaSuccess;
  k_alloc_pages<<<grid_for(need, 256, c.num_sms), 256, 0, s>>>(
      need, c.cfg.page_size, c.full, c.swa, c.mapping, c.mapping_len, out_full, out_swa,
      c.err_word);
  k_advance<<<1, 1, 0, s>>>(c.full, c.swa, need / c.cfg.page_size);
  return cudaGetLastError();
}

static size_t bitmap_bytes(int64_t cap) { return (size_t)((cap + 1 + 31) / 32) * 4; }

cudaError_t launch_merge_sorted(Ctx &c, bool full_pool, cudaStream_t s) {
  PoolDev p = full_pool ? c.full : c.swa;
  size_t smem = bitmap_bytes(p.cap);
  cudaFuncSetAttribute(k_merge_sorted, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_merge_sorted<<<1, 1024, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_release(Ctx &c, const int64_t *idx, int64_t n, bool do_full,
                           int64_t expect_full, int64_t expect_swa, cudaStream_t s) {
  size_t smem = bitmap_bytes(c.full.cap > c.swa.cap ? c.full.cap : c.swa.cap);
  cudaFuncSetAttribute(k_release, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_release<<<1, 1024, smem, s>>>(idx, n, do_full ? 1 : 0, c.cfg.page_size, c.full, c.swa,
                                   c.mapping, c.mapping_len, c.cfg.need_sort, expect_full,
                                   expect_swa, c.err_word);
  return cudaGetLastError();
}

cudaError_t launch_evict(Ctx &c, int bs, const int32_t *rt, int64_t rt_stride,
                         const int64_t *req_idx, const int64_t *pre, int64_t *evicted,
                         const int64_t *prot, int interval, int radix, cudaStream_t s) {
  if (bs == 0) return cudaSuccess;
  const bool paged = c.swa.ring_cost == 0;
  k_evict_plan<<<bs, 256, 0, s>>>(bs, rt, rt_stride, req_idx, pre, evicted, prot, c.lookback,
                                  c.cfg.page_size, interval, radix, c.mapping, c.mapping_len,
                                  paged, c.ev, c.err_word);
  const size_t smem = paged ? bitmap_bytes(c.swa.cap) : 0;
  cudaFuncSetAttribute(k_evict_apply, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_evict_apply<<<bs, 1024, smem, s>>>(bs, rt, rt_stride, req_idx, c.cfg.page_size, c.swa,
                                       c.mapping, c.mapping_len, c.ev, c.cfg.need_sort,
                                       c.err_word);
  k_evict_commit<<<1, 256, 0, s>>>(bs, evicted, c.swa, c.ev, c.cfg.need_sort);
  return cudaGetLastError();
}

cudaError_t launch_translate_for_kernel(const int64_t *v2p, int64_t n_pages, const int64_t *virt,
                                       int64_t n, int64_t ps, int64_t multiplier, int64_t *out,
                                       int32_t *err, int sms, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  k_translate_for_kernel<<<grid_for(n, 256, sms > 0 ? sms : 148), 256, 0, s>>>(
      v2p, n_pages, virt, n, ps, ps * multiplier, out, err);
  return cudaGetLastError();
}

cudaError_t launch_translate(Ctx &c, const int64_t *full_loc, int64_t n, int64_t *swa_loc,
                             cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  k_translate<<<grid_for(n, 256, c.num_sms), 256, 0, s>>>(full_loc, n, c.mapping,
                                                          c.mapping_len, swa_loc, c.err_word);
  return cudaGetLastError();
}

}  // namespace swa
