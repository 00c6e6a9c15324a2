// Chunked-prefill (extend) attention on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA): bf16 KV with D = 64 or 128, or E4M3 KV with D = 128
// (per-layer pools or the page-major envelope), any GQA group G up to 128,
// page size 16..64 (a power of two).
//
// Method: "SWA in SGLang" design note - the chunk's queries at positions
// pre..seq-1 attend causally; sliding layers see the last Wx+1 keys, full
// layers every earlier key; a per-head sink joins the denominator.
//
// GB300 design (persistent: one CTA per SM loops over work items; 10 warps,
// 12 for E4M3 KV, warp-specialised; TMEM and barriers set up once per CTA, barrier phases
// following running counts, so that no role waits for the others at an item
// boundary):
//   * an item is two Q tiles of up to 128 rows, each floor(128/G) consecutive
//     query tokens x the G query heads of one KV head (the tile's last 128 mod
//     G rows, if any, are unused rows whose weights are zero), so every K/V
//     tile it loads feeds two QK^T and two PV products;
//   * warp 9 finds each item (a warp-wide prefix count over the requests),
//     derives its key tiles and hands it to the other roles through a
//     two-slot ring in shared memory (so that their loops carry no per-item
//     arithmetic); it loads the Q tiles with TMA (box {64 dims, G heads,
//     floor(128/G) tokens}) into three rotating buffers - a buffer is released by
//     the epilogue that staged its tile's output through it, so the next
//     item's first tile is loaded while the current item still computes -
//     looks up page rows 32 page slots at a time with its lanes, a batch
//     ahead, and from one lane streams K and V through a
//     two-stage ring with TMA: one 3-D box
//     {64 dims, 1 head, ps rows} per page and 64-dim block of D, 128-byte swizzle,
//     completion counted on "full" mbarriers, slots returned on "empty" ones;
//   * warp 8 (one lane) issues tcgen05.mma: S_i = Q_i K^T into TMEM columns
//     [128 i, 128 i + 128) and O_i += P_i V into columns [256 + D i, ...),
//     with P_i read from TMEM where it overwrote S_i, and tcgen05.commit for
//     every hand-off;
//   * warps 0-3 and 4-7 are the softmax groups of Q tile 0 and 1: each thread
//     owns one row (one TMEM lane), reads its S row, masks only the key tiles
//     (64-key chunks on windowed layers) that straddle a window or causal
//     edge, and keeps a lazily rescaled running maximum (O in TMEM is rescaled
//     only when the maximum grew by more than 2^8), writes P as packed bf16
//     (f16 for E4M3 KV) pairs back to TMEM and signals the MMA lane; after the
//     item's last tile it normalises O (with the sink) and stores its output
//     rows, while the tensor core already computes the next item's first S;
//   * E4M3 KV only: warps 10 and 11 convert the K/V rows and the Q tiles to
//     f16 (below, at the kernel).
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
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "swa_internal.h"

namespace swa {
namespace {

constexpr int kRows = 128;                   // rows of one Q tile (M)
constexpr int kKeys = 128;                   // keys per K/V tile
constexpr int kThreads = 320;                // 8 softmax warps + MMA warp + load warp
constexpr int kThreadsF8 = 384;              // ... + 2 warps converting E4M3 K/V and Q to f16
constexpr int kBlock = kRows * 64 * 2;       // one 64-column block of a 128-row tile (16 KB)
// A 128-row (or 128-key) tile of D bf16 columns: D / 64 blocks of
// [128 rows][128 B] with the 128-byte swizzle.
template <int D>
struct Geo {
  static constexpr int kTileBytes = kRows * D * 2;
  static constexpr int kOffQ = 0;                  // Q buffers 0, 1, 2
  static constexpr int kOffK = 3 * kTileBytes;     // K stage 0, 1
  static constexpr int kOffV = 5 * kTileBytes;     // V stage 0, 1
  static constexpr int kOffBars = 7 * kTileBytes;  // mbarriers
  static constexpr int kCPR = D / 8;               // 16-byte chunks of a row
};
constexpr uint32_t kTmemCols = 512;
constexpr long kSpinLimit = 1L << 24;
constexpr float kRescaleGap = 8.f;           // log2 units: rescale O when the max grows more
constexpr float kSumCap = 65536.f;           // a chunk's weight sum that forces a maximum pass

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
  int32_t *err;
  // E4M3 KV only: the layer's K and V rows (row r of head h at r * row_bytes +
  // h * D bytes) and their dequantisation scales.
  const uint8_t *k8, *v8;
  int64_t row_bytes;
  float k_scale, v_scale;
};

// ------------------------------------------------------------------ PTX ---
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
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

// Pulls a box of the tensor into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Bulk tensor store of a box from shared memory (tracked by the issuing
// thread's bulk async-group), its commit, and the waits for the group's
// shared-memory reads (the source may be reused) or for its completion.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, int c0, int c1, int c2,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// tcgen05 shared-memory matrix descriptor: start >> 4 at [0,14), leading byte
// offset >> 4 at [16,30), stride byte offset >> 4 at [32,46), version 1 at
// [46,48), layout 2 (128-byte swizzle) at [61,64).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: D f32, A and B bf16 (type 1 at [7,10) and
// [10,13)) or both f16 (type 0), A K-major, B major bit 16, N >> 3 at [17,23),
// M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major, bool f16 = false) {
  return (1u << 4) | (f16 ? 0u : (1u << 7) | (1u << 10)) | ((b_mn_major ? 1u : 0u) << 16) |
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

__device__ __forceinline__ int64_t key_lo(int kind, int window, int64_t p) {
  if (kind == SWA_LAYER_FULL) return 0;
  if (kind == SWA_LAYER_SLIDING) return p - window > 0 ? p - window : 0;
  return (p / window) * window;
}

// E4M3 KV: four E4M3 values (bytes 0..3 of w) to two f16 pairs, low byte in
// the low half (exact: E4M3 is a subset of f16); a bf16 pair to an f16 pair
// (queries; round to nearest); a 16-byte read-only global load.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x));
  __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 ld_nc16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
// P = exp2(...) packed as the MMA's A type: bf16 pairs, or f16 pairs (E4M3 KV,
// whose operands are f16), and back.
template <bool kF16>
__device__ __forceinline__ uint32_t pack_p(float a, float b) {
  if constexpr (kF16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}
template <bool kF16>
__device__ __forceinline__ float2 unpack_p(uint32_t x) {
  if constexpr (kF16) return __half22float2(*reinterpret_cast<const __half2 *>(&x));
  else return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x));
}

// (row r, 16-byte chunk c) of a 128-row tile of D bf16 columns stored as D / 64
// blocks of [128 rows][128 B] with the 128-byte swizzle: the layout in which
// TMA writes a Q tile and reads an output tile.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * kBlock + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Shared memory (offsets from a 1024-byte aligned base): Geo<D>, then the
// mbarriers.  FULLQ / QFREE belong to the three Q buffers, IFULL / IEMPTY to
// the two-slot ring through which the producer hands items to the others,
// STAGED to each softmax group's output tile staged for its bulk store, QCONV
// (E4M3 KV) to the Q buffers converted to f16 in place.
enum { B_FULLK = 0, B_EMPTYK = 2, B_FULLV = 4, B_EMPTYV = 6, B_SDONE = 8, B_PREADY = 10,
       B_ODONE = 12, B_FULLQ = 14, B_QFREE = 17, B_IFULL = 20, B_IEMPTY = 22, B_STAGED = 24,
       B_DRAIN = 26, B_QCONV = 27, B_COUNT = 30 };
constexpr int kItemReaders = 9;              // the 8 softmax warps and the MMA lane (+2 converters)

// A work item: 2T consecutive query tokens of request b (clipped to the end
// of its chunk, qend), starting at token q0 and key position pfirst, with its
// key tiles (filled in by the producer, item_geo); b < 0 marks the end of the
// CTA's items.
struct Item {
  int b, n_tok, n_tiles;                // request; tokens; key tiles
  int64_t q0, qend, pfirst, kt0;        // first key tile kt0 (128-aligned)
};
struct ItemGeo {
  int64_t n_tok, k_lo, k_hi, kt0;   // tokens; key range; first key tile (128-aligned)
  int n_tiles;
};
__device__ __forceinline__ ItemGeo item_geo(const TcParams &P, const Item &it, int T2) {
  ItemGeo g;
  g.n_tok = min((int64_t)T2, it.qend - it.q0);
  g.k_lo = key_lo(P.kind, P.window, it.pfirst);
  g.k_hi = it.pfirst + g.n_tok - 1;
  g.kt0 = (g.k_lo / kKeys) * kKeys;
  g.n_tiles = (int)((g.k_hi - g.kt0) / kKeys + 1);
  return g;
}

// Warp-collective: the item numbered tau (the latest tokens first) as a
// request and its first token, or false past the last item.  The lanes take
// 32 requests at a time and count their items with a prefix sum.
__device__ __forceinline__ bool find_item(const TcParams &P, int64_t tau, int T2, int lane,
                                          Item &it) {
  int64_t acc = 0;
  for (int b0 = 0; b0 < P.bs; b0 += 32) {
    const int bb = b0 + lane;
    int64_t lo = 0, hi = 0, n = 0;
    if (bb < P.bs) {
      lo = P.qo_indptr[bb];
      hi = P.qo_indptr[bb + 1];
      n = (hi - lo + T2 - 1) / T2;
    }
    int64_t incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, bb < P.bs && tau < acc + incl);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const int64_t local = (tau - acc - __shfl_sync(0xffffffffu, incl - n, l)) * T2;
      it.b = b0 + l;
      it.q0 = __shfl_sync(0xffffffffu, lo, l) + local;
      it.qend = __shfl_sync(0xffffffffu, hi, l);
      it.pfirst = P.pre[it.b] + local;
      return true;
    }
    acc += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;
}

// The page that holds key position pos of a request, in two steps so that
// the load's latency can overlap other work: page_record() loads its record -
// the request's req_to_token entry (full layers: rt_row) or its entry in the
// request's SWA plan (hdr = the plan header h0, h2, h3, pages = the page list)
// - or -1 when the plan holds none; page_first_row() turns a record into the
// page's first row in the layer's K/V view, with the range and evicted-slot
// checks (an offending page reads as page 0).
__device__ __forceinline__ int32_t page_record(bool full, int ps_shift, const int32_t *rt_row,
                                               int64_t h0, int64_t h2, int64_t h3,
                                               const int32_t *pages, int64_t pos) {
  if (full) return rt_row[pos];
  const int64_t k = (pos >> ps_shift) - h2;
  return (pos >= h0 && k >= 0 && k < h3) ? pages[k] : -1;
}
__device__ __forceinline__ int32_t page_first_row(bool full, int ps_shift, int64_t page_stride,
                                                  int64_t max_page, int32_t rec, int32_t *err) {
  int64_t page = full ? (rec >= 0 ? rec >> ps_shift : -1) : rec;
  if (!full && page == 0) set_error(err, SWA_DEVERR_WINDOW_EVICTED);
  if (page < 0 || page > max_page) {
    set_error(err, SWA_DEVERR_RANGE);
    page = 0;
  }
  return (int32_t)(page * page_stride);
}

// kWin: a sliding-window or chunked layer, whose key tiles mostly straddle a
// window or causal edge; its softmax decides the masks per 64-key chunk and
// skips chunks outside every row's range.  Full layers (kWin false) mask per
// key tile, which keeps their loop - the one that sets the pace of the long
// causal rows - smaller in the instruction cache.
//
// kF8: E4M3 KV.  Two more warps (10, 11) read the K/V rows with plain loads
// (through their own page lookups), convert them to f16 (exact) into the
// stage buffers, and convert each Q tile to f16 in place once TMA has landed
// it; the MMAs then run with f16 operands, P is packed as f16, the K scale
// joins the softmax scale and the V scale the output normalisation.
template <int kD, bool kWin, bool kF8>
__global__ void __launch_bounds__(kF8 ? kThreadsF8 : kThreads, 1)
    k_extend_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                TcParams P) {
  using Gm = Geo<kD>;
  static_assert(!kF8 || kD == 128, "E4M3 KV: D = 128");
  constexpr int kTileBytes = Gm::kTileBytes, kOffQ = Gm::kOffQ, kOffK = Gm::kOffK;
  constexpr int kOffV = Gm::kOffV, kCPR = Gm::kCPR;
  extern __shared__ char smem_raw[];
  char *smem = reinterpret_cast<char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Gm::kOffBars);
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ Item s_item[2];
  __shared__ int32_t s_rows[2][32];        // page rows of 32 page slots, double-buffered

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y;
  const int G = P.G;
  const int T = kRows / G;                 // tokens per Q tile
  const int TG = T * G;                    // rows of a Q tile in use (128 unless G divides it not)
  const int T2 = 2 * T;                    // tokens per item
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
      mbar_init(bar(B_FULLK + i), kF8 ? 64 : 1);
      mbar_init(bar(B_EMPTYK + i), 1);
      mbar_init(bar(B_FULLV + i), kF8 ? 64 : 1);
      mbar_init(bar(B_EMPTYV + i), 1);
      mbar_init(bar(B_SDONE + i), 1);
      mbar_init(bar(B_PREADY + i), kRows);
      mbar_init(bar(B_ODONE + i), 1);
      mbar_init(bar(B_IFULL + i), 1);
      mbar_init(bar(B_IEMPTY + i), kItemReaders + (kF8 ? 2 : 0));
      mbar_init(bar(B_STAGED + i), kRows);
    }
    for (int j = 0; j < 3; ++j) {
      mbar_init(bar(B_FULLQ + j), 1);
      mbar_init(bar(B_QFREE + j), kRows);
      mbar_init(bar(B_QCONV + j), 64);
    }
    mbar_init(bar(B_DRAIN), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  constexpr uint32_t kIdS = idesc_f16(128, 128, false, kF8);
  constexpr uint32_t kIdO = idesc_f16(128, kD, true, kF8);

  // Persistent: the producer takes items blockIdx.x, blockIdx.x + gridDim.x,
  // ... and publishes each one; the other roles follow the published order.
  // Every barrier phase follows a running count - key tiles (tg), items (nd)
  // or Q tiles (u = 2 nd + tile, buffer u % 3) - so the rings run on across
  // items and no role waits for another at an item boundary.
  // Producer only, for the abort path: running counts of the K / V tiles and
  // Q tiles whose loads were issued.
  int k_issued = 0, v_issued = 0, q_issued = 0;

  if (warp == 9) {
    // ===================== producer: items, Q tiles, K/V pages =====================
    const int64_t max_page = P.pool_rows / P.ps - 1;
    const int ppt = kKeys / P.ps;            // pages per key tile (at most 8)
    int n_pub = 0, tg = 0;
    bool ok = true;
    auto wait_all = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, &s_abort));
    };
    // Item n goes to ring slot n & 1 once its readers have copied item n - 2.
    auto publish = [&](const Item &it) {
      const int slot = n_pub & 1;
      if (n_pub >= 2 && !wait_all(bar(B_IEMPTY + slot), ((n_pub >> 1) - 1) & 1)) return false;
      if (lane == 0) {
        s_item[slot] = it;
        mbar_arrive(bar(B_IFULL + slot));
      }
      __syncwarp();
      ++n_pub;
      return true;
    };
    // Q tile u of the CTA (tokens from tok on) into buffer u % 3, once the
    // epilogue of the tile that used the buffer before has released it.
    auto load_q = [&](int u, int64_t tok) {
      const int j = u % 3, f = u / 3;
      if (f >= 1 && !wait_all(bar(B_QFREE + j), (f - 1) & 1)) return false;
      if (lane == 0) {
        mbar_expect_tx(bar(B_FULLQ + j), (uint32_t)(TG * 128 * (kD / 64)));
        for (int h = 0; h < kD / 64; ++h)
          tma_load_3d(sb + kOffQ + j * kTileBytes + h * kBlock, &tmQ, h * 64, kvh * G, (int)tok,
                      bar(B_FULLQ + j));
      }
      __syncwarp();
      q_issued = u + 1;
      return true;
    };
    for (int item = blockIdx.x; ok && item < P.items_upper; item += gridDim.x) {
      Item it;
      if (!find_item(P, (int64_t)P.items_upper - 1 - item, T2, lane, it)) continue;
      const ItemGeo g = item_geo(P, it, T2);
      it.n_tok = (int)g.n_tok;
      it.n_tiles = g.n_tiles;
      it.kt0 = g.kt0;
      if (!(ok = publish(it))) break;
      if constexpr (kF8) {
        // E4M3 KV: the converter warps read K and V; only the Q tiles here.
        const int u0 = 2 * (n_pub - 1);
        if (!(ok = load_q(u0, it.q0))) break;
        if (lane == 0 && it.q0 + T < it.qend)
          for (int h = 0; h < kD / 64; ++h) tma_prefetch_3d(&tmQ, h * 64, kvh * G, (int)(it.q0 + T));
        if (!(ok = load_q(u0 + 1, it.q0 + T))) break;
        continue;
      }
      const int64_t pg0 = g.kt0 >> P.ps_shift;
      const int n_pg = (int)((g.k_hi >> P.ps_shift) - pg0 + 1);
      const int n_slots = g.n_tiles * ppt;
      const bool full_layer = P.kind == SWA_LAYER_FULL;
      const int32_t *rt_row = full_layer ? P.rt + P.req_idx[it.b] * P.rt_stride : nullptr;
      const int32_t *pages = full_layer ? nullptr : P.plan.pages + (int64_t)it.b * P.plan.max_pages;
      int64_t h0 = 0, h2 = 0, h3 = 0;
      if (!full_layer) {
        const int32_t *hdr = P.plan.hdr + it.b * 4;
        h0 = hdr[0];
        h2 = hdr[2];
        h3 = hdr[3];
      }
      auto first_row = [&](int32_t rec) {
        return page_first_row(full_layer, P.ps_shift, P.page_stride, max_page, rec, P.err);
      };
      // Every page slot of every key tile is loaded, so the stage buffers never
      // hold uninitialised bytes and need no clearing: slots outside the key
      // range load the item's first in-range page instead, whose values are
      // finite and get zero weight.  (Not page 0: mapping 0 marks an evicted
      // SWA slot, which attention must never read.)
      const int32_t row_lo =
          first_row(page_record(full_layer, P.ps_shift, rt_row, h0, h2, h3, pages, g.k_lo));
      // Records of the 32 page slots 32 k .. 32 k + 31, lane i for slot 32 k + i
      // (in range: -2 marks a slot outside the key range).
      auto batch_records = [&](int k) {
        const int i = 32 * k + lane;
        const int64_t pos0 = (pg0 + i) << P.ps_shift;
        const int64_t pos = pos0 > g.k_lo ? pos0 : g.k_lo;
        return i < n_pg && pos <= g.k_hi && pos0 + P.ps > g.k_lo
                   ? page_record(full_layer, P.ps_shift, rt_row, h0, h2, h3, pages, pos)
                   : -2;
      };
      auto batch_rows = [&](int32_t rec) { return rec == -2 ? row_lo : first_row(rec); };
      // Rows of the item's first 32 slots go to s_rows[0]; the records of the
      // next 32 are loaded now and turned into rows a batch later, so that a
      // batch's lookups overlap the previous batch's 32 / ppt tiles.
      s_rows[0][lane] = batch_rows(batch_records(0));
      int32_t rec_next = n_slots > 32 ? batch_records(1) : -2;
      __syncwarp();
      const int u0 = 2 * (n_pub - 1);
      if (!(ok = load_q(u0, it.q0))) break;
      // The second tile's buffer is released later (by the previous item's
      // first epilogue); its rows are pulled into L2 meanwhile.
      if (lane == 0 && it.q0 + T < it.qend)
        for (int h = 0; h < kD / 64; ++h) tma_prefetch_3d(&tmQ, h * 64, kvh * G, (int)(it.q0 + T));
      for (int t = 0; t < g.n_tiles && ok; ++t) {
        const int Tr = tg + t;               // the CTA's running tile count
        const int s = Tr & 1;
        const int i0 = t * ppt;              // the tile's first page slot (ppt divides 32)
        if (i0 > 0 && (i0 & 31) == 0) {
          s_rows[(i0 >> 5) & 1][lane] = batch_rows(rec_next);
          rec_next = i0 + 32 < n_slots ? batch_records((i0 >> 5) + 1) : -2;
          __syncwarp();
        }
        // One lane waits for the stages and issues the loads.
        int good = 1;
        if (lane == 0) {
          const int32_t *rows = &s_rows[(i0 >> 5) & 1][i0 & 31];
          for (int kv = 0; kv < 2 && good; ++kv) {
            if (Tr >= 2 &&
                !(good = mbar_wait(bar((kv ? B_EMPTYV : B_EMPTYK) + s), ((Tr >> 1) - 1) & 1,
                                   &s_abort)))
              break;
            const uint32_t full = bar((kv ? B_FULLV : B_FULLK) + s);
            const uint32_t dst = sb + (kv ? kOffV : kOffK) + s * kTileBytes;
            mbar_expect_tx(full, (uint32_t)kTileBytes);
            for (int i = 0; i < ppt; ++i)
              for (int h = 0; h < kD / 64; ++h)
                tma_load_3d(dst + h * kBlock + i * P.ps * 128, kv ? &tmV : &tmK, h * 64, kvh,
                            rows[i], full);
            if (kv) v_issued = Tr + 1;
            else k_issued = Tr + 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, good, 0) != 0;
        if (ok && t == 0) ok = load_q(u0 + 1, it.q0 + T);
        __syncwarp();
      }
      tg += g.n_tiles;
    }
    if (ok) {
      Item end;
      end.b = -1;
      end.n_tok = end.n_tiles = 0;
      end.q0 = end.qend = end.pfirst = end.kt0 = 0;
      publish(end);
    }
  } else if (warp == 8) {
    // ===================== MMA issue (one lane) =====================
    // Order per tile t: O0(t), S0(t+1), O1(t), S1(t+1) - softmax group 0 works
    // on tile t+1 while the tensor core runs O1(t) and S1(t+1), and group 1
    // likewise one slot later.  An item's first S0 is issued as soon as its Q
    // tile and first K tile have landed, while the groups still drain the
    // previous item's O.
    // Shared-memory descriptors built once per buffer and stage: a K step only
    // advances the 14-bit address field by (byte offset >> 4), which cannot
    // carry out of the field (shared addresses stay below 256 KB), so each
    // product's descriptors are one add from these.
    const uint64_t dq0 = smem_desc(sb + kOffQ, 16, 1024);   // buffer j: + j * kTileBytes >> 4
    const uint64_t dk0 = smem_desc(sb + kOffK, 16, 1024);
    const uint64_t dk1 = smem_desc(sb + kOffK + kTileBytes, 16, 1024);
    const uint64_t dv0 = smem_desc(sb + kOffV, kBlock, 1024);
    const uint64_t dv1 = smem_desc(sb + kOffV + kTileBytes, kBlock, 1024);
    auto issue_s = [&](int i, uint64_t qd, int Tr) {   // Tr: running tile count (stage)
      const uint64_t kd = (Tr & 1) ? dk1 : dk0;
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint64_t off16 = ((ks >> 2) * kBlock + (ks & 3) * 32) >> 4;
        mma_ss(tmem + i * 128, qd + off16, kd + off16, kIdS, ks > 0);
      }
      tc_commit(bar(B_SDONE + i));
    };
    auto issue_o = [&](int i, int t, int Tr) {   // t: tile of the item, Tr: running count
      const uint64_t vd = (Tr & 1) ? dv1 : dv0;
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks)
        mma_ts(tmem + 256 + i * kD, tmem + i * 128 + ks * 8, vd + (uint64_t)(ks * 16 * 128 >> 4),
               kIdO, (t > 0 || ks > 0) ? 1u : 0u);
    };
    if (lane == 0) {
      int tg = 0, nd = 0;
      for (bool ok = true; ok;) {
        const int slot = nd & 1;
        if (!mbar_wait(bar(B_IFULL + slot), (nd >> 1) & 1, &s_abort)) break;
        const Item it = s_item[slot];
        mbar_arrive(bar(B_IEMPTY + slot));
        if (it.b < 0) break;
        const int n_tiles = it.n_tiles;
        const int u0 = 2 * nd;
        const uint64_t qa = dq0 + (uint64_t)((u0 % 3) * kTileBytes >> 4);
        const uint64_t qb = dq0 + (uint64_t)(((u0 + 1) % 3) * kTileBytes >> 4);
        if (!mbar_wait(bar(B_FULLK + (tg & 1)), (tg >> 1) & 1, &s_abort)) break;
        if (!mbar_wait(bar((kF8 ? B_QCONV : B_FULLQ) + u0 % 3), (u0 / 3) & 1, &s_abort)) break;
        tc_fence_after();
        issue_s(0, qa, tg);
        if (!mbar_wait(bar((kF8 ? B_QCONV : B_FULLQ) + (u0 + 1) % 3), ((u0 + 1) / 3) & 1,
                       &s_abort))
          break;
        tc_fence_after();
        issue_s(1, qb, tg);
        tc_commit(bar(B_EMPTYK + (tg & 1)));
        for (int t = 0; t < n_tiles; ++t) {
          const int Tr = tg + t;
          const int s = Tr & 1, s1 = (Tr + 1) & 1;
          const bool more = t + 1 < n_tiles;
          if (!(ok = mbar_wait(bar(B_FULLV + s), (Tr >> 1) & 1, &s_abort))) break;
          if (!(ok = mbar_wait(bar(B_PREADY + 0), Tr & 1, &s_abort))) break;
          tc_fence_after();
          issue_o(0, t, Tr);
          if (more) {
            if (!(ok = mbar_wait(bar(B_FULLK + s1), ((Tr + 1) >> 1) & 1, &s_abort))) break;
            tc_fence_after();
            issue_s(0, qa, Tr + 1);
          } else {
            tc_commit(bar(B_ODONE + 0));
          }
          if (!(ok = mbar_wait(bar(B_PREADY + 1), Tr & 1, &s_abort))) break;
          tc_fence_after();
          issue_o(1, t, Tr);
          tc_commit(bar(B_EMPTYV + s));
          if (more) {
            issue_s(1, qb, Tr + 1);
            tc_commit(bar(B_EMPTYK + s1));
          } else {
            tc_commit(bar(B_ODONE + 1));
          }
        }
        tg += n_tiles;
        ++nd;
      }
    }
  } else if (warp >= 10) {
    // ============ converters (E4M3 KV only): Q, K and V to f16 ============
    // Per item: Q tile 0 (in place), then per key tile K and V into their
    // stages, Q tile 1 after the first key tile.  Each K or V tile's 16-byte
    // loads are issued before the wait for its stage, so their latency
    // overlaps that wait (the converters run ahead of the tensor core).
    const int ct = tid - kThreads;            // 0 .. 63
    const int64_t max_page = P.pool_rows / P.ps - 1;
    const int ppt = kKeys / P.ps;
    auto wait_all = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, &s_abort));
    };
    auto convert_q = [&](int u) {
      const int j = u % 3;
      if (!wait_all(bar(B_FULLQ + j), (u / 3) & 1)) return false;
      char *buf = smem + kOffQ + j * kTileBytes;
#pragma unroll 4
      for (int i = ct; i < kTileBytes / 16; i += 64) {
        uint4 *q16 = reinterpret_cast<uint4 *>(buf + i * 16);
        uint4 v = *q16;
        v.x = bf16x2_to_f16x2(v.x);
        v.y = bf16x2_to_f16x2(v.y);
        v.z = bf16x2_to_f16x2(v.z);
        v.w = bf16x2_to_f16x2(v.w);
        *q16 = v;
      }
      fence_async_smem();   // read by the tensor core (the async proxy)
      mbar_arrive(bar(B_QCONV + j));
      return true;
    };
    int tg = 0, nd = 0;
    for (bool ok = true; ok;) {
      const int slot = nd & 1;
      if (!wait_all(bar(B_IFULL + slot), (nd >> 1) & 1)) break;
      const Item it = s_item[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_IEMPTY + slot));
      if (it.b < 0) break;
      const int64_t k_lo = key_lo(P.kind, P.window, it.pfirst);
      const int64_t k_hi = it.pfirst + it.n_tok - 1;
      const int64_t pg0 = it.kt0 >> P.ps_shift;
      const int n_pg = (int)((k_hi >> P.ps_shift) - pg0 + 1);
      const bool full_layer = P.kind == SWA_LAYER_FULL;
      const int32_t *rt_row = full_layer ? P.rt + P.req_idx[it.b] * P.rt_stride : nullptr;
      const int32_t *pages = full_layer ? nullptr : P.plan.pages + (int64_t)it.b * P.plan.max_pages;
      int64_t h0 = 0, h2 = 0, h3 = 0;
      if (!full_layer) {
        const int32_t *hdr = P.plan.hdr + it.b * 4;
        h0 = hdr[0];
        h2 = hdr[2];
        h3 = hdr[3];
      }
      auto first_row = [&](int32_t rec) {
        return page_first_row(full_layer, P.ps_shift, P.page_stride, max_page, rec, P.err);
      };
      // Slots outside the key range read the first in-range page (finite
      // values, zero weight), as in the bf16 path.
      const int32_t row_lo =
          first_row(page_record(full_layer, P.ps_shift, rt_row, h0, h2, h3, pages, k_lo));
      auto batch_rows = [&](int k) {   // lane i: row of page slot 32 k + i
        const int i = 32 * k + lane;
        const int64_t pos0 = (pg0 + i) << P.ps_shift;
        const int64_t pos = pos0 > k_lo ? pos0 : k_lo;
        return i < n_pg && pos <= k_hi && pos0 + P.ps > k_lo
                   ? first_row(page_record(full_layer, P.ps_shift, rt_row, h0, h2, h3, pages, pos))
                   : row_lo;
      };
      int32_t rows = batch_rows(0);
      int cur_batch = 0;
      // The 16 chunks of 16 E4M3 dims this thread converts of key tile t of
      // K (kv = 0) or V: chunk idx = i * 64 + ct is key idx / 8, dims
      // 16 (idx % 8) .. + 15.
      auto load_tile = [&](int t, int kv, uint4 (&w)[16]) {
        const int i0 = t * ppt;
        if ((i0 >> 5) != cur_batch) {
          cur_batch = i0 >> 5;
          rows = batch_rows(cur_batch);
        }
        const uint8_t *src = (kv ? P.v8 : P.k8) + kvh * kD + (ct & 7) * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = i * 8 + (ct >> 3);                 // key of the tile
          const int32_t prow = __shfl_sync(0xffffffffu, rows, (i0 & 31) + (e >> P.ps_shift));
          w[i] = ld_nc16(src + (int64_t)(prow + (e & (P.ps - 1))) * P.row_bytes);
        }
      };
      auto store_tile = [&](int Tr, int kv, const uint4 (&w)[16]) {
        const int st = Tr & 1;
        if (Tr >= 2 && !wait_all(bar((kv ? B_EMPTYV : B_EMPTYK) + st), ((Tr >> 1) - 1) & 1))
          return false;
        char *dst = smem + (kv ? kOffV : kOffK) + st * kTileBytes;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = i * 8 + (ct >> 3), c = (ct & 7) * 2;   // f16 16-byte chunks c, c + 1
          uint4 a, b;
          e4m3x4_to_f16x4(w[i].x, a.x, a.y);
          e4m3x4_to_f16x4(w[i].y, a.z, a.w);
          e4m3x4_to_f16x4(w[i].z, b.x, b.y);
          e4m3x4_to_f16x4(w[i].w, b.z, b.w);
          *reinterpret_cast<uint4 *>(dst + tile_off(e, c)) = a;
          *reinterpret_cast<uint4 *>(dst + tile_off(e, c + 1)) = b;
        }
        fence_async_smem();   // read by the tensor core (the async proxy)
        mbar_arrive(bar((kv ? B_FULLV : B_FULLK) + st));
        return true;
      };
      const int u0 = 2 * nd;
      uint4 w[16];
      load_tile(0, 0, w);
      if (!(ok = convert_q(u0))) break;
      for (int t = 0; t < it.n_tiles && ok; ++t) {
        if (!(ok = store_tile(tg + t, 0, w))) break;
        load_tile(t, 1, w);
        if (!(ok = store_tile(tg + t, 1, w))) break;
        if (t + 1 < it.n_tiles) load_tile(t + 1, 0, w);
        if (t == 0) ok = convert_q(u0 + 1);
      }
      tg += it.n_tiles;
      ++nd;
    }
  } else {
    // ===================== softmax group i (warps 4i .. 4i+3) =====================
    const int grp = warp >> 2;
    const int r = tid & 127;                    // row of Q tile grp = TMEM lane
    const int tr = grp * T + r / G, g = r % G;  // token offset in the item, head
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + grp * 128 + lane_off;
    const uint32_t tO = tmem + 256 + grp * kD + lane_off;
    const int Hq = P.hkv * G;
    // The row's sink logit in log2 units (its head is fixed for the CTA's life).
    const float sg2 = P.sinks ? P.sinks[kvh * G + g] * 1.4426950408889634f : -INFINITY;
    int tg = 0, nd = 0, n_staged = 0;
    for (;;) {
      const int slot = nd & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_IFULL + slot), (nd >> 1) & 1, &s_abort)))
        break;
      const Item it = s_item[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_IEMPTY + slot));
      if (it.b < 0) break;
      const bool row_valid = r < TG && tr < it.n_tok;
      const int64_t p_row = it.pfirst + tr;
      const int64_t lo_row = key_lo(P.kind, P.window, p_row);
      float m_run = -INFINITY, l_run = 0.f;
      bool alive = true;
      for (int t = 0; t < it.n_tiles; ++t) {
        // Warp-uniform outcome: the TMEM loads below are warp-collective.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SDONE + grp), (tg + t) & 1, &s_abort))) {
          alive = false;
          break;
        }
        tc_fence_after();
        const int64_t j0 = it.kt0 + (int64_t)t * kKeys;
        const bool edge = !row_valid || j0 < lo_row || j0 + kKeys - 1 > p_row;
        // Key e of this tile counts iff lo_row <= j0 + e <= p_row (edge tiles only).
        const int e_lo = edge ? (int)max((int64_t)0, min((int64_t)kKeys, lo_row - j0)) : 0;
        const int e_hi = edge ? (row_valid ? (int)max((int64_t)-1, min((int64_t)kKeys - 1, p_row - j0))
                                           : -1)
                              : kKeys - 1;
        // Keys outside this row's range read as -inf where some row of the warp
        // has a window or causal edge (per tile on full layers, per 64-key
        // chunk on windowed ones): the max and the exponentials below then
        // need no per-key test.
        const bool masked = !kWin && __any_sync(0xffffffffu, edge);
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
        const float sc = kF8 ? P.scale_log2 * P.k_scale : P.scale_log2;
        const uint64_t sc2 = f2pack(sc, sc);
        uint64_t acc2[2] = {0ull, 0ull};   // running pair sums (two chains)
  #pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
          const int c0 = cb * 64;
          // On windowed layers a chunk outside every row's range (a window's
          // far side, the causal future) has all-zero weights: P = 0 and
          // nothing accumulates.
          if (kWin && __all_sync(0xffffffffu, e_hi < c0 || e_lo > c0 + 63)) {
            uint32_t zero[32];
  #pragma unroll
            for (int e = 0; e < 32; ++e) zero[e] = 0u;
            TC_ST32(tS + cb * 32, zero);
            continue;
          }
          uint32_t rr[64];
          TC_LD32(tS + cb * 64, rr);        // two loads in flight before one wait
          TC_LD32(tS + cb * 64 + 32, (rr + 32));
          tc_wait_ld();
          if (kWin ? __any_sync(0xffffffffu, e_lo > c0 || e_hi < c0 + 63) : masked)
            mask_in_place(rr, cb);
          // The reference maximum m_run moves only when needed: for a row's
          // first chunk (no reference yet), or when the chunk's weights against
          // the current reference sum past kSumCap (some score outgrew the
          // reference by more than log2 kSumCap - 6); otherwise the chunk's
          // maximum is never computed.  A chunk whose sum overflowed is
          // recomputed once against the raised reference.
          bool redo = __any_sync(0xffffffffu, m_run == -INFINITY);
          uint32_t pk[32];
          uint64_t c2[2];   // this chunk's pair sums
  #pragma unroll 1
          for (int pass = 0;; ++pass) {
            if (redo) {
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
                    const float2 f = unpack_p<kF8>(pp[e]);
                    pp[e] = pack_p<kF8>(f.x * corr, f.y * corr);
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
            }
            const float mu = m_run == -INFINITY ? 0.f : m_run;
            const uint64_t nmu2 = f2pack(-mu, -mu);
            // P = exp2(scale*s - m) as packed bf16 pairs, written over the S
            // columns already consumed (64-key chunk cb -> columns [32 cb, 32 cb + 32)).
            c2[0] = c2[1] = 0ull;
  #pragma unroll
            for (int e = 0; e < 32; ++e) {
              float t0, t1;
              f2unpack(fma2(f2pack(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1])), sc2, nmu2),
                       t0, t1);
              const float a0 = ex2(t0);
              const float a1 = ex2(t1);
              c2[e & 1] = add2(c2[e & 1], f2pack(a0, a1));
              pk[e] = pack_p<kF8>(a0, a1);
            }
            if (pass == 1) break;
            float s0, s1, s2, s3;
            f2unpack(c2[0], s0, s1);
            f2unpack(c2[1], s2, s3);
            redo = __any_sync(0xffffffffu, (s0 + s1) + (s2 + s3) > kSumCap);
            if (!redo) break;
          }
          acc2[0] = add2(acc2[0], c2[0]);
          acc2[1] = add2(acc2[1], c2[1]);
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
      if (!alive) break;
      // ---- epilogue ----
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_ODONE + grp), nd & 1, &s_abort))) break;
      tc_fence_after();
      const float mr = m_run == -INFINITY ? 0.f : m_run;
      const float mfin = fmaxf(mr, sg2);
      const float rsc = exp2f(mr - mfin);
      const float denom = l_run * rsc + (P.sinks ? exp2f(sg2 - mfin) : 0.f);
      const float f = (denom > 0.f ? rsc / denom : 0.f) * (kF8 ? P.v_scale : 1.f);
      // The output rows go through shared memory (this tile's Q buffer:
      // every product that read it has completed by ODONE).  On windowed
      // layers, whose items are short, a tile whose rows are all tokens of
      // the item is staged in the TMA layout and written by one bulk tensor
      // store; otherwise (full layers; a ragged tile at the end of a
      // request's chunk) the warps store the valid rows.
      const int jq = (2 * nd + grp) % 3;
      char *qbuf = smem + kOffQ + jq * kTileBytes;
      const bool whole = kWin && grp * T + T <= it.n_tok;
      char *stage = qbuf + (warp & 3) * 32 * (kD * 2);
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
          char *dst = whole ? qbuf + tile_off(r, c)
                            : stage + lane * (kD * 2) + ((c ^ (lane & (kCPR - 1))) << 4);
          *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (whole) {
        // Generic-proxy writes made visible to the bulk copy, then handed to
        // the group's first thread, which issues the store and releases the
        // buffer once the copy has read it.
        fence_async_smem();
        mbar_arrive(bar(B_STAGED + grp));
        if ((tid & 127) == 0) {
          if (mbar_wait(bar(B_STAGED + grp), n_staged & 1, &s_abort)) {
            for (int h = 0; h < kD / 64; ++h)
              tma_store_3d(&tmO, h * 64, kvh * G, (int)(it.q0 + grp * T),
                           sb + kOffQ + jq * kTileBytes + h * kBlock);
            bulk_commit();
            bulk_wait_read();
          }
        }
        ++n_staged;
      } else {
        __syncwarp();
#pragma unroll 4
        for (int idx = lane; idx < 32 * kCPR; idx += 32) {
          const int i = idx / kCPR, c = idx % kCPR;
          const int rw = (warp & 3) * 32 + i;     // row of Q tile grp
          const int trw = grp * T + rw / G;
          if (rw < TG && trw < it.n_tok) {
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + i * (kD * 2) +
                                                             ((c ^ (i & (kCPR - 1))) << 4));
            *reinterpret_cast<uint4 *>(P.out + ((it.q0 + trw) * Hq + kvh * G + rw % G) * kD +
                                       c * 8) = v;
          }
        }
        // The buffer's next contents arrive by TMA (the async proxy): order
        // these accesses before it.
        fence_async_smem();
      }
      mbar_arrive(bar(B_QFREE + jq));
      tg += it.n_tiles;
      ++nd;
    }
  }
  // The output stores complete before the CTA exits.
  if (kWin && warp < 8 && (tid & 127) == 0) bulk_wait_all();
  // Every role has left its loop: s_abort is final.
  __syncthreads();
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
      for (int j = 0; j < 3; ++j) {
        const int nf = q_issued > j ? (q_issued - 1 - j) / 3 + 1 : 0;   // fills of buffer j
        if (nf) mbar_drain(bar(B_FULLQ + j), (nf - 1) & 1);
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

template <int D, bool kWin, bool kF8>
cudaError_t launch_d(dim3 grid, const LayerInfo &L, const CUtensorMap &tmq, const CUtensorMap &tmo,
                     const TcParams &P, cudaStream_t s) {
  const size_t smem = 1024 + Geo<D>::kOffBars + B_COUNT * 8;
  static_assert(1024 + Geo<128>::kOffBars + B_COUNT * 8 + sizeof(Item) * 2 + 2 * 32 * 4 + 16 <=
                    227 * 1024,
                "shared memory of a CTA");
  cudaError_t e =
      cudaFuncSetAttribute(k_extend_tc<D, kWin, kF8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  k_extend_tc<D, kWin, kF8><<<grid, kF8 ? kThreadsF8 : kThreads, smem, s>>>(L.tmk, L.tmv, tmq, tmo, P);
  return cudaGetLastError();
}

bool tc_extend_supported(const Ctx &c, int layer) {
  const bool f8 = c.cfg.kv_dtype == SWA_DTYPE_E4M3;
  if (!c.layers[layer].tma || (c.cfg.kv_dtype != SWA_DTYPE_BF16 && !f8) ||
      (c.cfg.head_dim != 64 && c.cfg.head_dim != 128) || (f8 && c.cfg.head_dim != 128) ||
      c.cfg.page_size > 64)
    return false;
  const int G = c.cfg.num_q_heads / c.layers[layer].hkv;
  return G >= 1 && G <= kRows;
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
  P.err = c.err_word;
  const bool f8 = c.cfg.kv_dtype == SWA_DTYPE_E4M3;
  P.k8 = reinterpret_cast<const uint8_t *>(L.addr.k);
  P.v8 = reinterpret_cast<const uint8_t *>(L.addr.v);
  P.row_bytes = L.addr.row_bytes;
  P.k_scale = a.k_scale;
  P.v_scale = a.v_scale;
  // Persistent: one CTA per SM (the KV heads share the SMs), each looping
  // over its items.
  const int per_head = std::max(1, (c.num_sms > 0 ? c.num_sms : 148) / L.hkv);
  dim3 grid(std::min(P.items_upper, per_head), L.hkv);
  // Q and the output as [nq][Hq][D] tensors, one box = one 128-row tile of a
  // KV head's G heads.
  CUtensorMap tmq, tmo;
  if (!make_qo_tensor_map(&tmq, a.q, a.nq, c.cfg.num_q_heads, c.cfg.head_dim, P.G) ||
      !make_qo_tensor_map(&tmo, a.out, a.nq, c.cfg.num_q_heads, c.cfg.head_dim, P.G))
    return cudaErrorInvalidValue;
  const bool win = L.kind != SWA_LAYER_FULL;
  if (f8)
    return win ? launch_d<128, true, true>(grid, L, tmq, tmo, P, s)
               : launch_d<128, false, true>(grid, L, tmq, tmo, P, s);
  if (c.cfg.head_dim == 64)
    return win ? launch_d<64, true, false>(grid, L, tmq, tmo, P, s)
               : launch_d<64, false, false>(grid, L, tmq, tmo, P, s);
  return win ? launch_d<128, true, false>(grid, L, tmq, tmo, P, s)
             : launch_d<128, false, false>(grid, L, tmq, tmo, P, s);
}

}  // namespace swa
