// Persistent, TMA-fed paged decode attention (bf16 or FP8-E4M3 KV, one head
// row of 128 or 256 bytes, GQA group G <= 16, page size 16..128).
//
// Method: "SWA in SGLang" design note - sliding layers read the window of
// Wx+1 keys through the per-batch SWA page table, full layers every key
// through req_to_token; a per-head sink joins the softmax denominator.
//
// GB300 design.  Decode streams K/V from HBM once, so the kernel is built to
// keep as many bytes in flight as shared memory allows:
//   * one CTA per SM takes work items (request, KV head, split of up to 1024
//     keys) from a global counter, so the stream never drains at a CTA
//     boundary and an SM that runs slow simply takes fewer items;
//   * warp 4 is the producer: its 32 lanes look up the page rows of the next
//     item in parallel, then lane 0 issues one TMA box {128 bytes of the head
//     row, 1 head, min(ps, 64) rows} per page and half-row into a ring of
//     kStages 64-key stages (~160 KB), counted on "full" mbarriers and
//     recycled through "empty" mbarriers;
//   * warps 0-3 consume: warp w owns keys 16w..16w+15 of each stage and runs
//     QK^T and PV on mma.sync.m16n8k16 (the G query heads are the M rows,
//     zero-padded to 16) with an online softmax in registers; FP8 rows are
//     widened to f16 by the warp that owns them, so no CTA barrier sits in
//     the stage loop;
//   * at the end of an item the four warps merge through shared memory; a
//     single-split item writes the output (with the sink), otherwise a
//     partial goes to the workspace and the last split to finish (atomic
//     ticket) merges all partials.
// Rows of a loaded page outside the item's key range get zero weight; pools
// are zero-initialised by the caller and the ring is zeroed at start, so
// every row the tensor cores read is finite.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include "split_merge.cuh"
#include "swa_internal.h"

namespace swa {
namespace {

constexpr int kTileKeys = 64;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kMaxSplitKeys = 8192;
constexpr int kMaxPg = kMaxSplitKeys / 16 + 2;   // page rows of one item (ps >= 16)
constexpr long kSpinLimit = 1L << 24;

struct Params {
  int kind, window, hkv, G, ps;
  int64_t page_stride;
  int64_t pool_rows;
  const int32_t *rt;
  int64_t rt_stride;
  const int64_t *req_idx;
  const int64_t *seq;
  int bs;
  PlanView plan;
  const __nv_bfloat16 *q;
  const float *sinks;
  float qk_scale_log2;
  float v_scale;
  __nv_bfloat16 *out;
  float *partials;
  int32_t *tickets;
  int32_t *work;         // [0] next item, [1] CTAs finished (reset by the last CTA)
  int max_splits;
  int split_keys;         // keys per work item (a multiple of the tile)
  int32_t *err;
};

template <int D, bool FP8>
struct Cfg {
  static constexpr int kEsz = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kEsz;             // stored bytes of one head row
  static constexpr int kBlocks = kRowBytes / 128;         // 128-byte column blocks per row
  static constexpr int kTile = kTileKeys * kRowBytes;     // K (or V) of one stage
  static constexpr int kStage = 2 * kTile;
  // Ring sized so that two CTAs share an SM (8 consumer warps per SM).
  static constexpr int kStages = (FP8 ? 32 : 64) * 1024 / kStage;
  static constexpr int kRing = kStages * kStage;
  static constexpr int kWidePerWarp = FP8 ? 2 * 16 * D * 2 : 0;   // f16 K,V of 16 rows
  static constexpr int kWide = kConsumers * kWidePerWarp;
  static constexpr int kQ = 16 * D * 2;
  static constexpr int kMergeO = kConsumers * 16 * (D + 4) * 4;
  static constexpr int kMergeML = 2 * kConsumers * 16 * 4;
  static constexpr int kOffWide = kRing;
  static constexpr int kOffQ = kOffWide + kWide;
  static constexpr int kOffMerge = kOffQ + kQ;
  static constexpr int kOffRows = kOffMerge + kMergeO + kMergeML;
  static constexpr int kOffBars = kOffRows + kMaxPg * 4;
  static constexpr int kBytes = kOffBars + 2 * kStages * 8 + 64;
  static_assert(kMergeO >= kMergeScratchBytes, "split merge scratch exceeds the merge buffers");
};

// ------------------------------------------------------------------ PTX ---
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  for (long i = 0; i < kSpinLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 1023) == 1023 && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
struct ConsumerSync {   // barrier 1 over the consumer warps
  __device__ void operator()() const { named_sync(1, kConsumers * 32); }
};
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// 16-bit tile of R rows x D columns stored as D/64 blocks of [R][128 B] with
// the 128-byte swizzle (the layout TMA writes); c = 16-byte chunk (8 elements).
template <int R>
__device__ __forceinline__ uint32_t t16(int r, int c) {
  return (uint32_t)((c >> 3) * (R * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Work item -> (b, kvh, split) through per-request split counts.
struct Item {
  int b, kvh, split, n_splits;
  int64_t k0, k1, lo;   // keys [k0, k1) of this split; lo = first key of the request's range
};

__device__ __forceinline__ int64_t key_lo(int kind, int window, int64_t p) {
  if (kind == SWA_LAYER_FULL) return 0;
  if (kind == SWA_LAYER_SLIDING) return p - window > 0 ? p - window : 0;
  return (p / window) * window;
}

__device__ __forceinline__ bool find_item(const Params &P, const int *s_pref, int idx, Item &it) {
  // s_pref[b] = items before request b (each request has n_splits * hkv items)
  int lo = 0, hi = P.bs;
  if (idx < 0 || idx >= s_pref[P.bs]) return false;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= idx) lo = mid; else hi = mid;
  }
  it.b = lo;
  const int local = idx - s_pref[lo];
  const int64_t p = P.seq[lo] - 1;
  it.lo = key_lo(P.kind, P.window, p);
  it.n_splits = (int)((p - it.lo + 1 + P.split_keys - 1) / P.split_keys);
  it.kvh = local % P.hkv;                 // heads of one split adjacent: rows shared in DRAM
  it.split = local / P.hkv;
  it.k0 = it.lo + (int64_t)it.split * P.split_keys;
  it.k1 = min(p + 1, it.k0 + P.split_keys);
  return true;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, 2)
    k_decode_tma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 Params P) {
  using C = Cfg<D, FP8>;
  constexpr bool F16 = FP8;
  extern __shared__ char smem_raw[];
  char *smem = reinterpret_cast<char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  int32_t *s_rows = reinterpret_cast<int32_t *>(smem + C::kOffRows);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
  __shared__ int s_pref[1025];
  __shared__ volatile int s_abort;
  __shared__ int s_last;
  __shared__ int s_item[32], s_tile[32];   // item / tile carried by each stage
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[C::kStages + s]); };

  // ---- item prefix over requests ----
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < P.bs; ++b) {
      s_pref[b] = acc;
      const int64_t p = P.seq[b] - 1;
      const int64_t lo = key_lo(P.kind, P.window, p);
      acc += (int)((p - lo + 1 + P.split_keys - 1) / P.split_keys) * P.hkv;
    }
    s_pref[P.bs] = acc;
    s_abort = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  for (int i = tid; i < C::kRing / 16; i += kThreads)
    reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  __syncthreads();

  const int n_items = s_pref[P.bs];
  const int G = P.G;
  const int Hq = P.hkv * G;

  if (warp == kConsumers) {
    // =========================== producer ===========================
    // Items come from a global counter (any idle SM takes the next one); each
    // stage is tagged with its item and tile so the consumers follow.
    const int rows_per_box = P.ps < kTileKeys ? P.ps : kTileKeys;
    const int64_t max_page = P.pool_rows / P.ps - 1;
    uint32_t g = 0;   // stage counter (used by lane 0)
    while (true) {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(P.work, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      Item it;
      const bool have = idx < n_items && !s_abort && find_item(P, s_pref, idx, it);
      if (!have) {
        if (lane == 0) {   // one stage tagged "no more work"
          const int s = g % C::kStages;
          if (g < (uint32_t)C::kStages ||
              mbar_wait(empty_bar(s), ((g / C::kStages) - 1) & 1, &s_abort)) {
            s_item[s] = -1;
            s_tile[s] = 0;
            mbar_arrive(full_bar(s));
          }
        }
        break;
      }
      const int64_t kt0 = (it.k0 / kTileKeys) * kTileKeys;
      const int n_tiles = (int)((it.k1 - 1 - kt0) / kTileKeys + 1);
      const int64_t pg0 = kt0 / P.ps;
      const int n_pg = (int)((it.k1 - 1) / P.ps - pg0 + 1);
      if (n_pg > kMaxPg || n_tiles > P.split_keys / kTileKeys + 1) {   // cannot happen for ps >= 16
        if (lane == 0) {
          set_error(P.err, SWA_DEVERR_RANGE);
          s_abort = 1;
        }
        break;
      }
      for (int i = lane; i < n_pg; i += 32) {
        const int64_t pos0 = (pg0 + i) * P.ps;
        const int64_t pos = pos0 > it.k0 ? pos0 : it.k0;
        int32_t row = -1;
        if (pos0 + P.ps > it.k0) {
          int64_t page;
          if (P.kind == SWA_LAYER_FULL) {
            page = P.rt[P.req_idx[it.b] * P.rt_stride + pos] / P.ps;
          } else {
            const int32_t *h = P.plan.hdr + it.b * 4;
            const int64_t k = pos / P.ps - h[2];
            page = (pos >= h[0] && k >= 0 && k < h[3])
                       ? P.plan.pages[(int64_t)it.b * P.plan.max_pages + k] : -1;
            if (page == 0) set_error(P.err, SWA_DEVERR_WINDOW_EVICTED);
          }
          if (page < 0 || page > max_page) {
            set_error(P.err, SWA_DEVERR_RANGE);
            page = 0;
          }
          row = (int32_t)(page * P.page_stride);
        }
        s_rows[i] = row;
      }
      __syncwarp();
      if (lane == 0) {
        for (int t = 0; t < n_tiles; ++t, ++g) {
          const int s = g % C::kStages;
          if (g >= (uint32_t)C::kStages &&
              !mbar_wait(empty_bar(s), ((g / C::kStages) - 1) & 1, &s_abort))
            break;
          s_item[s] = idx;
          s_tile[s] = t;
          const int64_t j0 = kt0 + (int64_t)t * kTileKeys;
          uint32_t bytes = 0;
          for (int64_t r0 = j0; r0 < j0 + kTileKeys; r0 += rows_per_box)
            if (r0 < it.k1 && r0 + rows_per_box > it.k0 && s_rows[r0 / P.ps - pg0] >= 0)
              bytes += (uint32_t)rows_per_box * C::kRowBytes * 2;
          mbar_expect_tx(full_bar(s), bytes);
          const uint32_t kd = sb + s * C::kStage, vd = kd + C::kTile;
          for (int64_t r0 = j0; r0 < j0 + kTileKeys; r0 += rows_per_box) {
            if (!(r0 < it.k1 && r0 + rows_per_box > it.k0)) continue;
            const int32_t prow = s_rows[r0 / P.ps - pg0];
            if (prow < 0) continue;
            const int row = prow + (int)(r0 % P.ps);
            const int rl = (int)(r0 - j0);
#pragma unroll
            for (int blk = 0; blk < C::kBlocks; ++blk) {
              const uint32_t off = blk * (kTileKeys * 128) + rl * 128;
              tma_load_3d(kd + off, &tmK, blk * (128 / C::kEsz), it.kvh, row, full_bar(s));
              tma_load_3d(vd + off, &tmV, blk * (128 / C::kEsz), it.kvh, row, full_bar(s));
            }
          }
        }
      }
      __syncwarp();
      if (s_abort) break;
    }
  } else {
    // =========================== consumers ===========================
    char *wide = smem + C::kOffWide + warp * C::kWidePerWarp;
    char *sq = smem + C::kOffQ;
    float *sm_o = reinterpret_cast<float *>(smem + C::kOffMerge);
    float *sm_m = sm_o + kConsumers * 16 * (D + 4);
    float *sm_l = sm_m + kConsumers * 16;
    const int g_row = lane >> 2, c4 = lane & 3;
    uint32_t g = 0;
    Item it;
    int64_t kt0 = 0;
    int n_tiles = 0;
    uint32_t qa[D / 16][4];
    float o[D / 8][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    while (true) {
      const int s = g % C::kStages;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(full_bar(s), (g / C::kStages) & 1, &s_abort);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      // Every lane acquires the completed phase itself (returns at once) so
      // the stage's tag and its TMA data are ordered for all of them.
      mbar_wait(full_bar(s), (g / C::kStages) & 1, &s_abort);
      const int idx = s_item[s], t = s_tile[s];
      if (idx < 0) break;
      if (t == 0) {
        // ---- a new item: its Q rows (padded to 16) into registers ----
        find_item(P, s_pref, idx, it);
        kt0 = (it.k0 / kTileKeys) * kTileKeys;
        n_tiles = (int)((it.k1 - 1 - kt0) / kTileKeys + 1);
        for (int i = tid; i < 16 * (D / 8); i += kConsumers * 32) {
          const int r = i / (D / 8), c = i % (D / 8);
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < G) {
            v = *reinterpret_cast<const uint4 *>(P.q + ((int64_t)it.b * Hq + it.kvh * G + r) * D + c * 8);
            if constexpr (F16) {
              const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&v);
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack2<true>(__bfloat162float(h[2 * e]), __bfloat162float(h[2 * e + 1]));
              v = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          *reinterpret_cast<uint4 *>(sq + t16<16>(r, c)) = v;
        }
        named_sync(1, kConsumers * 32);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int c = ks * 2 + (lane >> 4);
          ldsm_x4(smem_u32(sq + t16<16>(r, c)), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
#pragma unroll
        for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
      }
      {
        const char *kt = smem + s * C::kStage;
        const char *vt = kt + C::kTile;
        uint32_t kaddr, vaddr;   // 16-bit tiles read by ldmatrix
        int rbase;
        if constexpr (FP8) {
          // Widen this warp's 16 rows of K and V (E4M3 -> f16, exact).
          for (int i = lane; i < 2 * 16 * (D / 16); i += 32) {
            const int kv = i / (16 * (D / 16));
            const int rem = i % (16 * (D / 16));
            const int r = rem / (D / 16), c = rem % (D / 16);
            const int rr = warp * 16 + r;
            const char *src = (kv ? vt : kt) + (c >> 3) * (kTileKeys * 128) + rr * 128 +
                              (((c & 7) ^ (rr & 7)) << 4);
            const uint4 raw = *reinterpret_cast<const uint4 *>(src);
            const __nv_fp8x2_storage_t *f = reinterpret_cast<const __nv_fp8x2_storage_t *>(&raw);
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(f[e], __NV_E4M3);
              w[e] = (uint32_t)hr.x | ((uint32_t)hr.y << 16);
            }
            char *dst = wide + kv * (16 * D * 2);
            *reinterpret_cast<uint4 *>(dst + t16<16>(r, 2 * c)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4 *>(dst + t16<16>(r, 2 * c + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
          }
          __syncwarp();
          kaddr = smem_u32(wide);
          vaddr = smem_u32(wide + 16 * D * 2);
          rbase = 0;
        } else {
          kaddr = smem_u32(kt);
          vaddr = smem_u32(vt);
          rbase = warp * 16;
        }
        // Two accumulators per 8-key block halve the dependent mma chain.
        float sc[2][4], sx[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] = sx[nt][e] = 0.f;
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            const int r = rbase + nt * 8 + (lane & 7);
            const int c = kk * 4 + (lane >> 3);
            uint32_t b0, b1, b2, b3;
            const uint32_t a = FP8 ? kaddr + t16<16>(r, c) : kaddr + t16<kTileKeys>(r, c);
            ldsm_x4(a, b0, b1, b2, b3);
            mma16816<F16>(sc[nt], qa[2 * kk], b0, b1);
            mma16816<F16>(sx[nt], qa[2 * kk + 1], b2, b3);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] += sx[nt][e];
        }
        const int64_t jw = kt0 + (int64_t)t * kTileKeys + warp * 16;
        float rm0 = -INFINITY, rm1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t j = jw + nt * 8 + 2 * c4 + (e & 1);
            float v = sc[nt][e] * P.qk_scale_log2;
            if (j < it.k0 || j >= it.k1) v = -INFINITY;
            sc[nt][e] = v;
          }
          rm0 = fmaxf(rm0, fmaxf(sc[nt][0], sc[nt][1]));
          rm1 = fmaxf(rm1, fmaxf(sc[nt][2], sc[nt][3]));
        }
        rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 1));
        rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 2));
        rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 1));
        rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 2));
        const float mn0 = fmaxf(m0, rm0), mn1 = fmaxf(m1, rm1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float corr0 = ex2(m0 - mu0), corr1 = ex2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sc[nt][0] = ex2(sc[nt][0] - mu0);
          sc[nt][1] = ex2(sc[nt][1] - mu0);
          sc[nt][2] = ex2(sc[nt][2] - mu1);
          sc[nt][3] = ex2(sc[nt][3] - mu1);
          ps0 += sc[nt][0] + sc[nt][1];
          ps1 += sc[nt][2] + sc[nt][3];
        }
        l0 = l0 * corr0 + ps0;
        l1 = l1 * corr1 + ps1;
        if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {   // a row maximum moved
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            o[n][0] *= corr0;
            o[n][1] *= corr0;
            o[n][2] *= corr1;
            o[n][3] *= corr1;
          }
        }
        uint32_t pa[4];
        pa[0] = pack2<F16>(sc[0][0], sc[0][1]);
        pa[1] = pack2<F16>(sc[0][2], sc[0][3]);
        pa[2] = pack2<F16>(sc[1][0], sc[1][1]);
        pa[3] = pack2<F16>(sc[1][2], sc[1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int r = rbase + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int c = dp * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          const uint32_t a = FP8 ? vaddr + t16<16>(r, c) : vaddr + t16<kTileKeys>(r, c);
          ldsm_x4_t(a, b0, b1, b2, b3);
          mma16816<F16>(o[2 * dp], pa, b0, b1);
          mma16816<F16>(o[2 * dp + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
      ++g;
      if (t != n_tiles - 1) continue;
      // ---- last tile of the item: merge the four warps ----
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      constexpr int OS = D + 4;
      if (c4 == 0) {
        sm_m[warp * 16 + g_row] = m0;
        sm_m[warp * 16 + g_row + 8] = m1;
        sm_l[warp * 16 + g_row] = l0;
        sm_l[warp * 16 + g_row + 8] = l1;
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        float *r0p = sm_o + (warp * 16 + g_row) * OS + n * 8 + 2 * c4;
        float *r1p = sm_o + (warp * 16 + g_row + 8) * OS + n * 8 + 2 * c4;
        r0p[0] = o[n][0];
        r0p[1] = o[n][1];
        r1p[0] = o[n][2];
        r1p[1] = o[n][3];
      }
      named_sync(1, kConsumers * 32);
      const bool single = it.n_splits == 1;
      const int pstride = part_stride(G, D);
      const int64_t bh = (int64_t)it.b * P.hkv + it.kvh;
      float *part = P.partials + (bh * P.max_splits + it.split) * pstride;
      for (int e = tid; e < G * D; e += kConsumers * 32) {
        const int gg = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, sm_m[w * 16 + gg]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
          const float f = ex2(sm_m[w * 16 + gg] - Mu);
          L += sm_l[w * 16 + gg] * f;
          A += sm_o[(w * 16 + gg) * OS + d] * f;
        }
        if (single) {
          float Mf = Mu, extra = 0.f;
          if (P.sinks) {
            const float sg = P.sinks[it.kvh * G + gg] * 1.4426950408889634f;
            Mf = fmaxf(Mu, sg);
            extra = ex2(sg - Mf);
          }
          const float r = ex2(Mu - Mf);
          P.out[((int64_t)it.b * Hq + it.kvh * G + gg) * D + d] =
              __float2bfloat16_rn(A * r * P.v_scale / (L * r + extra));
        } else {
          part[gg * D + d] = A;
          if (d == 0) {
            part[G * D + 2 * gg] = Mu;
            part[G * D + 2 * gg + 1] = L;
          }
        }
      }
      if (!single) {
        __threadfence();
        named_sync(1, kConsumers * 32);
        if (tid == 0) s_last = atomicAdd(&P.tickets[bh], 1) == it.n_splits - 1;
        named_sync(1, kConsumers * 32);
        if (s_last) {
          __threadfence();
          merge_split_partials<D, kConsumers * 32, 1>(
              P.partials + bh * P.max_splits * pstride, it.n_splits, G,
              P.sinks ? P.sinks + it.kvh * G : nullptr, P.v_scale,
              P.out + ((int64_t)it.b * Hq + it.kvh * G) * D, P.tickets + bh, sm_o, tid,
              ConsumerSync());
        }
      }
      named_sync(1, kConsumers * 32);   // merge buffers and Q tile free for the next item
    }
  }
  // The last CTA to leave resets the work counter for the next launch.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.work + 1, 1) == (int)gridDim.x - 1) {
      P.work[0] = 0;
      P.work[1] = 0;
      __threadfence();
    }
  }
  if (s_abort && tid == 0) set_error(P.err, SWA_DEVERR_RANGE);
}

template <int D, bool FP8>
cudaError_t launch_t(Ctx &c, const LayerInfo &L, const Params &P, cudaStream_t s) {
  using C = Cfg<D, FP8>;
  const int smem = C::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_decode_tma<D, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k_decode_tma<D, FP8><<<2 * c.num_sms, kThreads, smem, s>>>(L.tmk, L.tmv, P);
  return cudaGetLastError();
}

int max_keys_of(const Ctx &c, int layer, int max_seq_len) {
  const LayerInfo &L = c.layers[layer];
  int64_t mk = max_seq_len;
  if (L.kind == SWA_LAYER_SLIDING && L.window + 1 < mk) mk = L.window + 1;
  if (L.kind == SWA_LAYER_CHUNKED && L.window < mk) mk = L.window;
  return (int)(mk < 1 ? 1 : mk);
}

}  // namespace

bool tma_decode_supported(const Ctx &c, int layer) {
  const LayerInfo &L = c.layers[layer];
  if (!L.tma) return false;
  if (c.cfg.max_batch > 1024) return false;
  const int G = c.cfg.num_q_heads / L.hkv;
  if (G < 1 || G > 16) return false;
  const int D = c.cfg.head_dim;
  if (c.cfg.kv_dtype == SWA_DTYPE_BF16) return D == 64 || D == 128;
  return c.cfg.kv_dtype == SWA_DTYPE_E4M3 && D == 128;
}

// Workspace: [work counters, 256 B][tickets][partials], the layout every
// attention family shares (the counters and tickets keep their place for
// layers of different shapes).
struct WsLayout {
  int split_keys, max_splits;
  size_t part_off, total;
};

static WsLayout ws_layout(const Ctx &c, int layer, int64_t nq, int max_seq_len) {
  const LayerInfo &L = c.layers[layer];
  const int G = c.cfg.num_q_heads / L.hkv;
  const int mk = max_keys_of(c, layer, max_seq_len);
  WsLayout w;
  w.split_keys = decode_split_keys(c.num_sms, nq, L.hkv, mk, c.cfg.page_size);
  if (w.split_keys > kMaxSplitKeys) w.split_keys = kMaxSplitKeys;
  w.max_splits = (mk + w.split_keys - 1) / w.split_keys;
  const size_t part = (size_t)nq * L.hkv * w.max_splits * part_stride(G, c.cfg.head_dim) * sizeof(float);
  w.part_off = ws_partials_off(c, nq);
  w.total = w.part_off + (part + 255) / 256 * 256;
  return w;
}

size_t tma_decode_ws_bytes(const Ctx &c, int layer, int64_t nq, int max_seq_len) {
  return ws_layout(c, layer, nq, max_seq_len).total;
}

cudaError_t launch_attn_decode_tma(Ctx &c, const AttnArgs &a, cudaStream_t s) {
  if (a.nq == 0) return cudaSuccess;
  const LayerInfo &L = c.layers[a.layer];
  const int G = c.cfg.num_q_heads / L.hkv;
  Params P;
  P.kind = L.kind;
  P.window = L.window;
  P.hkv = L.hkv;
  P.G = G;
  P.ps = c.cfg.page_size;
  P.page_stride = (int64_t)P.ps * (L.addr.blocks ? L.addr.blocks : 1);
  P.pool_rows = (L.in_full ? c.cfg.size_full : c.cfg.size_swa) + c.cfg.page_size;
  P.rt = a.rt;
  P.rt_stride = a.rt_stride;
  P.req_idx = a.req_idx;
  P.seq = a.seq;
  P.bs = a.bs;
  P.plan = a.plan;
  P.q = static_cast<const __nv_bfloat16 *>(a.q);
  P.sinks = a.sinks;
  const bool fp8 = c.cfg.kv_dtype == SWA_DTYPE_E4M3;
  P.qk_scale_log2 = a.scale * 1.4426950408889634f * (fp8 ? a.k_scale : 1.f);
  P.v_scale = fp8 ? a.v_scale : 1.f;
  P.out = static_cast<__nv_bfloat16 *>(a.out);
  const WsLayout w = ws_layout(c, a.layer, a.nq, a.max_seq_len);
  P.split_keys = w.split_keys;
  P.max_splits = w.max_splits;
  P.work = static_cast<int32_t *>(a.ws);
  P.partials = reinterpret_cast<float *>(static_cast<char *>(a.ws) + w.part_off);
  P.tickets = reinterpret_cast<int32_t *>(static_cast<char *>(a.ws) + 256);
  P.err = c.err_word;
  if (fp8) return launch_t<128, true>(c, L, P, s);
  if (c.cfg.head_dim == 128) return launch_t<128, false>(c, L, P, s);
  return launch_t<64, false>(c, L, P, s);
}

}  // namespace swa
