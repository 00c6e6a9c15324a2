// Chunked-prefill (extend) attention on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 KV in the per-layer layout, D = 64 or 128,
// GQA group G in {8, 16}, page size 16..64 (a power of two).
//
// Method: "SWA in SGLang" design note - the chunk's queries at positions
// pre..seq-1 attend causally; sliding layers see the last Wx+1 keys, full
// layers every earlier key; a per-head sink joins the denominator.
//
// GB300 design (persistent: one CTA per SM loops over work items; 10 warps,
// warp-specialised; TMEM and barriers set up once per CTA, barrier phases
// following the CTA's running tile count across items):
//   * an item is two 128-row Q tiles, each (128/G) consecutive query tokens
//     x the G query heads of one KV head, so every K/V tile it loads feeds two
//     QK^T and two PV products;
//   * all threads gather the Q rows once (cp.async) while the page rows are
//     looked up; then warp 9, from one lane,
//     streams K and V through a two-stage ring with TMA: one 3-D box
//     {64 dims, 1 head, ps rows} per page and 64-dim block of D, 128-byte swizzle,
//     completion counted on "full" mbarriers, slots returned on "empty" ones;
//   * warp 8 (one lane) issues tcgen05.mma: S_i = Q_i K^T into TMEM columns
//     [128 i, 128 i + 128) and O_i += P_i V into columns [256 + D i, ...),
//     with P_i read from TMEM where it overwrote S_i, and tcgen05.commit for
//     every hand-off;
//   * warps 0-3 and 4-7 are the softmax groups of Q tile 0 and 1: each thread
//     owns one row (one TMEM lane), reads its S row, masks only the key tiles
//     that straddle a window or causal edge, and keeps a lazily rescaled
//     running maximum (O in TMEM is rescaled only when the maximum grew by more
//     than 2^8), writes P as packed bf16 pairs back to TMEM and signals the
//     MMA lane; after the last tile it normalises O (with the sink) and stores
//     its output row.
// KV pools are zero-initialised by the caller (as the pages' pools are), so
// rows of a loaded page outside the query's key range hold finite values and
// their zero softmax weight cancels them exactly; page slots of a key tile
// outside the range load an in-range page of the same request for the same
// reason.
// Every mbarrier wait has a poll limit; on expiry the kernel sets
// SWA_DEVERR_TIMEOUT, every role leaves its loop, the TMA loads and tensor-core
// products already issued are waited for, and the TMEM is released.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "swa_internal.h"

namespace swa {
namespace {

constexpr int kRows = 128;                   // rows of one Q tile (M)
constexpr int kKeys = 128;                   // keys per K/V tile
constexpr int kThreads = 320;                // 8 softmax warps + MMA warp + load warp
constexpr int kBlock = kRows * 64 * 2;       // one 64-column block of a 128-row tile (16 KB)
// A 128-row (or 128-key) tile of D bf16 columns: D / 64 blocks of
// [128 rows][128 B] with the 128-byte swizzle.
template <int D>
struct Geo {
  static constexpr int kTileBytes = kRows * D * 2;
  static constexpr int kOffQ = 0;                  // Q0, Q1
  static constexpr int kOffK = 2 * kTileBytes;     // K stage 0, 1
  static constexpr int kOffV = 4 * kTileBytes;     // V stage 0, 1
  static constexpr int kOffRows = 6 * kTileBytes;  // int32 page rows [max_pages]
  static constexpr int kCPR = D / 8;               // 16-byte chunks of a row
};
constexpr uint32_t kTmemCols = 512;
constexpr long kSpinLimit = 1L << 24;
constexpr float kRescaleGap = 8.f;           // log2 units: rescale O when the max grows more

struct TcParams {
  int kind, window, hkv, G, ps, ps_shift;
  int64_t page_stride;   // rows between consecutive pages of the layer's view
  int64_t pool_rows;
  const int32_t *rt;
  int64_t rt_stride;
  const int64_t *req_idx;
  const int64_t *pre;
  const int64_t *qo_indptr;
  int bs;
  int items_upper;
  PlanView plan;
  const __nv_bfloat16 *q;
  const float *sinks;
  float scale_log2;
  __nv_bfloat16 *out;
  int max_pages;
  int32_t *err;
};

// ------------------------------------------------------------------ PTX ---
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
  int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
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
// Bounded wait for the phase of the given parity.  Gives up (returns false)
// after the poll limit or when another role has already aborted.
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
// Bounded wait used only after an abort, for work that completes on its own
// (issued TMA loads, committed tensor-core products): it ignores the flag.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  for (long i = 0; i < kSpinLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return;
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// tcgen05 shared-memory matrix descriptor: start >> 4 at [0,14), leading byte
// offset >> 4 at [16,30), stride byte offset >> 4 at [32,46), version 1 at
// [46,48), layout 2 (128-byte swizzle) at [61,64).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: D f32, A and B bf16, A K-major, B major
// bit 16, N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// A operand read from tensor memory (P), B from shared memory (V).
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}

#define TC_LD32(taddr, r)                                                                       \
  asm volatile(                                                                                 \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"  \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),          \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),          \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])           \
      : "r"(taddr))

#define TC_ST32(taddr, r)                                                                       \
  asm volatile(                                                                                 \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"   \
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"     \
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),          \
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),         \
        "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),     \
        "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),     \
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]))

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
// The SFU's base-2 exponential (flushes denormal results to zero, which only
// affects weights below 2^-126 relative to the row maximum).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// Paired fp32 arithmetic (one instruction for two lanes of values) and a
// three-input maximum: the softmax warps are bound by instruction issue, so
// halving the instructions per score element is what speeds them up.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// (row r, 16-byte chunk c in 0..15) of a 128 x 128 bf16 tile stored as two
// 64-column blocks of [128 rows][128 B] with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * kBlock + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ int64_t key_lo(int kind, int window, int64_t p) {
  if (kind == SWA_LAYER_FULL) return 0;
  if (kind == SWA_LAYER_SLIDING) return p - window > 0 ? p - window : 0;
  return (p / window) * window;
}

// Shared memory (offsets from a 1024-byte aligned base): Geo<D>.
enum { B_FULLK = 0, B_EMPTYK = 2, B_FULLV = 4, B_EMPTYV = 6, B_SDONE = 8, B_PREADY = 10,
       B_ODONE = 12, B_DRAIN = 13, B_COUNT = 14 };

template <int kD>
__global__ void __launch_bounds__(kThreads, 1)
    k_extend_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                TcParams P) {
  using Gm = Geo<kD>;
  constexpr int kTileBytes = Gm::kTileBytes, kOffQ = Gm::kOffQ, kOffK = Gm::kOffK;
  constexpr int kOffV = Gm::kOffV, kOffRows = Gm::kOffRows, kCPR = Gm::kCPR;
  extern __shared__ char smem_raw[];
  char *smem = reinterpret_cast<char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  int32_t *s_rows = reinterpret_cast<int32_t *>(smem + kOffRows);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffRows + ((P.max_pages * 4 + 7) & ~7));
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int64_t s_q0, s_qend, s_pfirst, s_req;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y;
  const int G = P.G;
  const int T = kRows / G;                 // tokens per Q tile
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  // ---- once per CTA: TMEM, barriers ----
  if (tid == 0) s_abort = 0;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_FULLK + i), 1);
      mbar_init(bar(B_EMPTYK + i), 1);
      mbar_init(bar(B_FULLV + i), 1);
      mbar_init(bar(B_EMPTYV + i), 1);
      mbar_init(bar(B_SDONE + i), 1);
      mbar_init(bar(B_PREADY + i), kRows);
    }
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  constexpr uint32_t kIdS = idesc_f16(128, 128, false);
  constexpr uint32_t kIdO = idesc_f16(128, kD, true);

  // Persistent: the CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...
  // Every barrier phase follows the CTA's running tile count tg0 (key tiles
  // of its earlier items) or item count n_done, so the rings run on across
  // items; each item ends with all roles joined (its Q tiles and TMEM free).
  int tg0 = 0, n_done = 0;
  // Producer only: running tile counts whose K / V loads were issued (tile T
  // arms phase T >> 1 of "full" barrier T & 1), so that an abort can wait for
  // the loads still in flight.
  int k_issued = 0, v_issued = 0;
  for (int item = blockIdx.x; item < P.items_upper; item += gridDim.x) {
  __syncthreads();   // every thread has read the previous item's fields
  // ---- work item: two Q tiles of one request, latest first ----
  if (tid == 0) {
    int64_t tau = (int64_t)P.items_upper - 1 - item, acc = 0;
    s_req = -1;
    for (int b = 0; b < P.bs; ++b) {
      const int64_t ext = P.qo_indptr[b + 1] - P.qo_indptr[b];
      const int64_t n = (ext + 2 * T - 1) / (2 * T);
      if (tau < acc + n) {
        const int64_t local = (tau - acc) * 2 * T;
        s_req = b;
        s_q0 = P.qo_indptr[b] + local;
        s_qend = P.qo_indptr[b + 1];
        s_pfirst = P.pre[b] + local;
        break;
      }
      acc += n;
    }
  }
  __syncthreads();
  if (s_req < 0) continue;
  const int b = (int)s_req;
  const int64_t q0 = s_q0, n_tok = min((int64_t)2 * T, s_qend - s_q0);
  const int64_t p_first = s_pfirst, p_last = p_first + n_tok - 1;
  const int64_t k_lo = key_lo(P.kind, P.window, p_first);
  const int64_t k_hi = p_last;
  const int64_t kt0 = (k_lo / kKeys) * kKeys;      // key tiles are 128-aligned
  const int n_tiles = (int)((k_hi - kt0) / kKeys + 1);
  const int64_t pg0 = kt0 / P.ps;
  const int n_pg = (int)(k_hi / P.ps - pg0 + 1);
  if (n_pg > P.max_pages || n_tiles * (kKeys / P.ps) > P.max_pages) {
    if (tid == 0) set_error(P.err, SWA_DEVERR_RANGE);
    continue;
  }

  // Q rows of both tiles, gathered by every thread (cp.async, zero fill past
  // the chunk); their latency overlaps the page-row lookups below.
  {
    const int Hq = P.hkv * G;
    for (int i = tid; i < 2 * kRows * kCPR; i += kThreads) {
      const int qt = i / (kRows * kCPR), rr = (i / kCPR) % kRows, c = i % kCPR;
      const int64_t tok = q0 + qt * T + rr / G;
      const bool ok = tok < s_qend && (qt * T + rr / G) < n_tok;
      const __nv_bfloat16 *src = P.q + ((ok ? tok : q0) * Hq + kvh * G + rr % G) * kD + c * 8;
      cp_async16(sb + kOffQ + qt * kTileBytes + tile_off(rr, c), src, ok);
    }
  }
  const int64_t max_page = P.pool_rows / P.ps - 1;
  // Every page slot of every key tile is loaded, so the stage buffers never
  // hold uninitialised bytes and need no clearing: slots outside the key
  // range (-1 here) load the item's first in-range page instead, whose
  // values are finite and get zero weight.  (Not page 0: mapping 0 marks an
  // evicted SWA slot, which attention must never read.)
  const int n_slots = n_tiles * (kKeys / P.ps);
  for (int i = tid; i < n_slots; i += kThreads) {
    const int64_t pos0 = (pg0 + i) * P.ps;
    const int64_t pos = pos0 > k_lo ? pos0 : k_lo;
    int64_t page = -2;                       // -2: outside the key range
    if (i < n_pg && pos <= k_hi && pos0 + P.ps > k_lo) {
      if (P.kind == SWA_LAYER_FULL) {
        page = P.rt[P.req_idx[b] * P.rt_stride + pos] / P.ps;
      } else {
        const int32_t *h = P.plan.hdr + b * 4;
        const int64_t k = pos / P.ps - h[2];
        page = (pos >= h[0] && k >= 0 && k < h[3]) ? P.plan.pages[(int64_t)b * P.plan.max_pages + k]
                                                   : -1;
        if (page == 0) set_error(P.err, SWA_DEVERR_WINDOW_EVICTED);
      }
      if (page < 0 || page > max_page) {
        set_error(P.err, SWA_DEVERR_RANGE);
        page = 0;
      }
    }
    s_rows[i] = page == -2 ? -1 : (int32_t)(page * P.page_stride);
  }
  const int slot_lo = (int)(k_lo / P.ps - pg0);   // first in-range slot
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  fence_async_smem();   // Q (written by cp.async) is read by the tensor core
  __syncthreads();
  tc_fence_after();

  if (warp == 9) {
    // ===================== producer: K/V pages =====================
    if (lane == 0) {
      const int pages_per_tile = kKeys / P.ps;
      for (int t = 0; t < n_tiles && !s_abort; ++t) {
        const int T = tg0 + t;             // the CTA's running tile count
        const int s = T & 1;
        for (int kv = 0; kv < 2; ++kv) {
          if (T >= 2 && !mbar_wait(bar((kv ? B_EMPTYV : B_EMPTYK) + s), ((T >> 1) - 1) & 1, &s_abort))
            break;
          const uint32_t full = bar((kv ? B_FULLV : B_FULLK) + s);
          mbar_expect_tx(full, (uint32_t)kTileBytes);   // every page slot is loaded
          if (kv) v_issued = T + 1;
          else k_issued = T + 1;
          const uint32_t dst = sb + (kv ? kOffV : kOffK) + s * kTileBytes;
          for (int i = 0; i < pages_per_tile; ++i) {
            const int pi = t * pages_per_tile + i;
            const int32_t row = s_rows[pi] >= 0 ? s_rows[pi] : s_rows[slot_lo];
            for (int h = 0; h < kD / 64; ++h)
              tma_load_3d(dst + h * kBlock + i * P.ps * 128, kv ? &tmV : &tmK, h * 64, kvh, row, full);
          }
        }
      }
    }
  } else if (warp == 8) {
    // ===================== MMA issue (one lane) =====================
    // Order per tile t: O0(t), S0(t+1), O1(t), S1(t+1) - softmax group 0 works
    // on tile t+1 while the tensor core runs O1(t) and S1(t+1), and group 1
    // likewise one slot later.
    // Shared-memory descriptors built once per tile and stage: a K step only
    // advances the 14-bit address field by (byte offset >> 4), which cannot
    // carry out of the field (shared addresses stay below 256 KB), so each
    // product's descriptors are one add from these.
    const uint64_t dq0 = smem_desc(sb + kOffQ, 16, 1024);
    const uint64_t dq1 = smem_desc(sb + kOffQ + kTileBytes, 16, 1024);
    const uint64_t dk0 = smem_desc(sb + kOffK, 16, 1024);
    const uint64_t dk1 = smem_desc(sb + kOffK + kTileBytes, 16, 1024);
    const uint64_t dv0 = smem_desc(sb + kOffV, kBlock, 1024);
    const uint64_t dv1 = smem_desc(sb + kOffV + kTileBytes, kBlock, 1024);
    auto issue_s = [&](int i, int T) {     // T: running tile count (stage)
      const uint64_t qd = i ? dq1 : dq0, kd = (T & 1) ? dk1 : dk0;
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint64_t off16 = ((ks >> 2) * kBlock + (ks & 3) * 32) >> 4;
        mma_ss(tmem + i * 128, qd + off16, kd + off16, kIdS, ks > 0);
      }
      tc_commit(bar(B_SDONE + i));
    };
    auto issue_o = [&](int i, int t, int T) {   // t: tile of the item, T: running count
      const uint64_t vd = (T & 1) ? dv1 : dv0;
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks)
        mma_ts(tmem + 256 + i * kD, tmem + i * 128 + ks * 8, vd + (uint64_t)(ks * 16 * 128 >> 4),
               kIdO, (t > 0 || ks > 0) ? 1u : 0u);
    };
    if (lane == 0 && mbar_wait(bar(B_FULLK + (tg0 & 1)), (tg0 >> 1) & 1, &s_abort)) {
      tc_fence_after();
      issue_s(0, tg0);
      issue_s(1, tg0);
      tc_commit(bar(B_EMPTYK + (tg0 & 1)));
      for (int t = 0; t < n_tiles; ++t) {
        const int T = tg0 + t;
        const int s = T & 1, s1 = (T + 1) & 1;
        const bool more = t + 1 < n_tiles;
        if (!mbar_wait(bar(B_FULLV + s), (T >> 1) & 1, &s_abort)) break;
        if (!mbar_wait(bar(B_PREADY + 0), T & 1, &s_abort)) break;
        tc_fence_after();
        issue_o(0, t, T);
        if (more) {
          if (!mbar_wait(bar(B_FULLK + s1), ((T + 1) >> 1) & 1, &s_abort)) break;
          tc_fence_after();
          issue_s(0, T + 1);
        }
        if (!mbar_wait(bar(B_PREADY + 1), T & 1, &s_abort)) break;
        tc_fence_after();
        issue_o(1, t, T);
        tc_commit(bar(B_EMPTYV + s));
        if (more) {
          issue_s(1, T + 1);
          tc_commit(bar(B_EMPTYK + s1));
        }
      }
    }
    if (lane == 0) tc_commit(bar(B_ODONE));
  } else {
    // ===================== softmax group i (warps 4i .. 4i+3) =====================
    const int grp = warp >> 2;
    const int r = tid & 127;                    // row of Q tile grp = TMEM lane
    const int tr = grp * T + r / G, g = r % G;  // token offset in the item, head
    const bool row_valid = tr < n_tok;
    const int64_t p_row = p_first + tr;
    const int64_t lo_row = key_lo(P.kind, P.window, p_row);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + grp * 128 + lane_off;
    const uint32_t tO = tmem + 256 + grp * kD + lane_off;
    float m_run = -INFINITY, l_run = 0.f;
    bool alive = true;
    for (int t = 0; t < n_tiles; ++t) {
      // Warp-uniform outcome: the TMEM loads below are warp-collective.
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SDONE + grp), (tg0 + t) & 1, &s_abort))) {
        alive = false;
        break;
      }
      tc_fence_after();
      const int64_t j0 = kt0 + (int64_t)t * kKeys;
      const bool edge = !row_valid || j0 < lo_row || j0 + kKeys - 1 > p_row;
      // Key e of this tile counts iff lo_row <= j0 + e <= p_row (edge tiles only).
      const int e_lo = edge ? (int)max((int64_t)0, min((int64_t)kKeys, lo_row - j0)) : 0;
      const int e_hi = edge ? (row_valid ? (int)max((int64_t)-1, min((int64_t)kKeys - 1, p_row - j0))
                                         : -1)
                            : kKeys - 1;
      // Interior tiles (no row of the warp at a window or causal edge) skip
      // the per-key masks entirely.
      const bool masked = __any_sync(0xffffffffu, edge);
      // Keys outside this row's range read as -inf (edge tiles only): the
      // max and the exponentials below then need no per-key test.
      auto mask_in_place = [&](uint32_t (&rr)[64], int cb) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int ee = cb * 64 + e;
          if (ee < e_lo || ee > e_hi) rr[e] = 0xff800000u;   // -inf
        }
      };
      // One pass over S, 64 keys at a time: each chunk's maximum is checked
      // against the running reference maximum m_run, which moves only when a
      // chunk exceeds it by more than kRescaleGap (weights stay below
      // 2^kRescaleGap meanwhile).  A move rescales what was accumulated
      // against the old reference - O of earlier tiles, the running sum and,
      // for the second chunk, the first chunk's P already in TMEM - before
      // this chunk's exponentials.  The 64-key loops stay rolled: one copy of
      // each body keeps the softmax code inside the instruction cache.
      const float sc = P.scale_log2;
      const uint64_t sc2 = f2pack(sc, sc);
      uint64_t acc2[2] = {0ull, 0ull};   // running pair sums (two chains)
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t rr[64];
        TC_LD32(tS + cb * 64, rr);        // two loads in flight before one wait
        TC_LD32(tS + cb * 64 + 32, (rr + 32));
        tc_wait_ld();
        if (masked) mask_in_place(rr, cb);
        // four independent chains of three-input maxima
        float m2[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 64; e += 2)
          m2[(e >> 1) & 3] = max3(m2[(e >> 1) & 3], __uint_as_float(rr[e]), __uint_as_float(rr[e + 1]));
        float cm = max3(m2[0], m2[1], fmaxf(m2[2], m2[3]));
        cm = cm == -INFINITY ? -INFINITY : cm * sc;
        // A row whose maximum is still -inf has accumulated exactly nothing
        // (every P so far was 0), so its first finite maximum needs no
        // rescale (factor 1): only moves of a finite maximum pay for one.
        float corr = 1.f;
        if (cm > m_run + kRescaleGap || (m_run == -INFINITY && cm != -INFINITY)) {
          corr = m_run == -INFINITY ? 1.f : exp2f(m_run - cm);
          m_run = cm;
        }
        if (__any_sync(0xffffffffu, corr != 1.f)) {
          if (t > 0) {
#pragma unroll 1
            for (int ob = 0; ob < kD / 32; ++ob) {
              uint32_t ro[32];
              TC_LD32(tO + ob * 32, ro);
              tc_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * corr);
              TC_ST32(tO + ob * 32, ro);
            }
          }
          if (cb == 1) {
            // the first chunk's P (32 columns of bf16 pairs) against the new reference
            uint32_t pp[32];
            tc_wait_st();
            TC_LD32(tS, pp);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&pp[e]);
              const float2 f = __bfloat1622float2(h);
              h = __floats2bfloat162_rn(f.x * corr, f.y * corr);
              pp[e] = *reinterpret_cast<uint32_t *>(&h);
            }
            TC_ST32(tS, pp);
          }
          float a0, a1, b0, b1;
          f2unpack(acc2[0], a0, a1);
          f2unpack(acc2[1], b0, b1);
          acc2[0] = f2pack(a0 * corr, a1 * corr);
          acc2[1] = f2pack(b0 * corr, b1 * corr);
          l_run *= corr;
        }
        const float mu = m_run == -INFINITY ? 0.f : m_run;
        const uint64_t nmu2 = f2pack(-mu, -mu);
        // P = exp2(scale*s - m) as packed bf16 pairs, written over the S
        // columns already consumed (64-key chunk cb -> columns [32 cb, 32 cb + 32)).
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float t0, t1;
          f2unpack(fma2(f2pack(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1])), sc2, nmu2),
                   t0, t1);
          const float a0 = ex2(t0);
          const float a1 = ex2(t1);
          acc2[e & 1] = add2(acc2[e & 1], f2pack(a0, a1));
          __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
          pk[e] = *reinterpret_cast<uint32_t *>(&h);
        }
        TC_ST32(tS + cb * 32, pk);
      }
      {
        float s0, s1, s2, s3;
        f2unpack(acc2[0], s0, s1);
        f2unpack(acc2[1], s2, s3);
        l_run += (s0 + s1) + (s2 + s3);
      }
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PREADY + grp));
    }
    // ---- epilogue ----
    if (alive && __all_sync(0xffffffffu, mbar_wait(bar(B_ODONE), n_done & 1, &s_abort))) {
      tc_fence_after();
      float sg2 = -INFINITY;
      if (P.sinks) sg2 = P.sinks[kvh * G + g] * 1.4426950408889634f;
      const float mr = m_run == -INFINITY ? 0.f : m_run;
      const float mfin = fmaxf(mr, sg2);
      const float rsc = exp2f(mr - mfin);
      const float denom = l_run * rsc + (P.sinks ? exp2f(sg2 - mfin) : 0.f);
      const float f = denom > 0.f ? rsc / denom : 0.f;
      const int Hq = P.hkv * G;
      // The warp's 32 output rows go through shared memory (the Q tile area:
      // every product that read it has completed by ODONE), so that the global
      // stores are whole 256-byte rows written by 16 consecutive lanes.
      char *stage = smem + kOffQ + grp * kTileBytes + (warp & 3) * 32 * (kD * 2);
#pragma unroll 1
      for (int cb = 0; cb < kD / 64; ++cb) {
        uint32_t rr[64];
        TC_LD32(tO + cb * 64, rr);
        TC_LD32(tO + cb * 64 + 32, (rr + 32));
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; e += 8) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(rr[e + 2 * k]) * f,
                                                     __uint_as_float(rr[e + 2 * k + 1]) * f);
            w[k] = *reinterpret_cast<uint32_t *>(&h);
          }
          const int c = (cb * 64 + e) >> 3;   // 16-byte chunk of the row
          *reinterpret_cast<uint4 *>(stage + lane * (kD * 2) + ((c ^ (lane & (kCPR - 1))) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      __syncwarp();
#pragma unroll 4
      for (int idx = lane; idx < 32 * kCPR; idx += 32) {
        const int i = idx / kCPR, c = idx % kCPR;
        const int rw = (warp & 3) * 32 + i;     // row of Q tile grp
        const int trw = grp * T + rw / G;
        if (trw < n_tok) {
          const uint4 v =
              *reinterpret_cast<const uint4 *>(stage + i * (kD * 2) + ((c ^ (i & (kCPR - 1))) << 4));
          *reinterpret_cast<uint4 *>(P.out + ((q0 + trw) * Hq + kvh * G + rw % G) * kD + c * 8) = v;
        }
      }
    }
  }
  // end of the item: all roles joined before its Q tiles and TMEM are reused
  tc_fence_before();
  __syncthreads();
  tg0 += n_tiles;
  ++n_done;
  if (s_abort) break;
  tc_fence_after();
  }
  if (s_abort) {
    // A role gave up a wait.  Loads and products already issued complete on
    // their own; wait for them before the shared memory and TMEM they write
    // are released.
    if (tid == 0) set_error(P.err, SWA_DEVERR_TIMEOUT);
    if (warp == 9 && lane == 0) {
      for (int i = 0; i < 2; ++i) {
        const int nk = (k_issued + 1 - i) >> 1, nv = (v_issued + 1 - i) >> 1;  // phases armed
        if (nk) mbar_drain(bar(B_FULLK + i), (nk - 1) & 1);
        if (nv) mbar_drain(bar(B_FULLV + i), (nv - 1) & 1);
      }
    }
    if (warp == 8 && lane == 0) {
      tc_commit(bar(B_DRAIN));   // tracks every product this thread issued
      mbar_drain(bar(B_DRAIN), 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

}  // namespace

template <int D>
cudaError_t launch_d(dim3 grid, size_t tail, const LayerInfo &L, const TcParams &P, cudaStream_t s) {
  const size_t smem = 1024 + Geo<D>::kOffRows + tail;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(k_extend_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_extend_tc<D><<<grid, kThreads, smem, s>>>(L.tmk, L.tmv, P);
  return cudaGetLastError();
}

bool tc_extend_supported(const Ctx &c, int layer) {
  if (!c.layers[layer].tma || c.cfg.kv_dtype != SWA_DTYPE_BF16 ||
      (c.cfg.head_dim != 64 && c.cfg.head_dim != 128) || c.cfg.page_size > 64)
    return false;
  const int G = c.cfg.num_q_heads / c.layers[layer].hkv;
  return G == 8 || G == 16;
}

size_t tc_extend_ws_bytes(const Ctx &, int, int64_t, int) { return 256; }

cudaError_t launch_attn_extend_tc(Ctx &c, const AttnArgs &a, cudaStream_t s) {
  if (a.nq == 0) return cudaSuccess;
  const LayerInfo &L = c.layers[a.layer];
  TcParams P;
  P.kind = L.kind;
  P.window = L.window;
  P.hkv = L.hkv;
  P.G = c.cfg.num_q_heads / L.hkv;
  P.ps = c.cfg.page_size;
  P.ps_shift = __builtin_ctz((unsigned)P.ps);
  P.page_stride = (int64_t)P.ps * (L.addr.blocks ? L.addr.blocks : 1);
  P.pool_rows = (L.in_full ? c.cfg.size_full : c.cfg.size_swa) + c.cfg.page_size;
  P.rt = a.rt;
  P.rt_stride = a.rt_stride;
  P.req_idx = a.req_idx;
  P.pre = a.pre;
  P.qo_indptr = a.qo_indptr;
  P.bs = a.bs;
  const int T2 = 2 * (kRows / P.G);
  P.items_upper = (int)((a.nq + T2 - 1) / T2 + a.bs);
  P.plan = a.plan;
  P.q = static_cast<const __nv_bfloat16 *>(a.q);
  P.sinks = a.sinks;
  P.scale_log2 = a.scale * 1.4426950408889634f;
  P.out = static_cast<__nv_bfloat16 *>(a.out);
  P.max_pages = a.max_seq_len / P.ps + kKeys / P.ps + 2;
  P.err = c.err_word;
  // Persistent: one CTA per SM (the KV heads share the SMs), each looping
  // over its items.
  const int per_head = std::max(1, (c.num_sms > 0 ? c.num_sms : 148) / L.hkv);
  dim3 grid(std::min(P.items_upper, per_head), L.hkv);
  const size_t tail = ((size_t)P.max_pages * 4 + 7) / 8 * 8 + B_COUNT * 8;
  if (c.cfg.head_dim == 64) return launch_d<64>(grid, tail, L, P, s);
  return launch_d<128>(grid, tail, L, P, s);
}

}  // namespace swa
