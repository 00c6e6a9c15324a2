// Chunked-prefill (extend) attention on the 5th-generation tensor cores
// (tcgen05 + TMEM), bf16 KV, D = 128, GQA group G in {8, 16}, page size >= 16.
//
// Method: "SWA in SGLang" design note - the chunk's queries at positions
// pre..seq-1 attend causally; sliding layers see the last Wx+1 keys, full
// layers every earlier key; a per-head sink joins the denominator.
//
// GB300 design.  In extend, QK^T and PV are dense tile contractions, so they
// run on tcgen05.mma (kind::f16, bf16 in, f32 accumulate in tensor memory):
//   * a CTA owns one 128-row Q tile = (128/G) query tokens x the G query heads
//     of one KV head (all rows share the KV head's keys);
//   * keys stream in tiles of 128 rows gathered through the index tables with
//     cp.async (16-byte chunks, 128-byte swizzle, double buffered);
//   * one thread issues S = Q K^T (M=128, N=128, K=128) into TMEM columns
//     0..127 and O += P V into columns 128..255; tcgen05.commit signals an
//     mbarrier;
//   * each of the 128 threads owns one TMEM lane = one row: it reads its S
//     row, applies the causal / window mask, runs the online softmax in
//     registers, writes its P row (bf16) to shared memory as the A operand of
//     the next MMA, and rescales its O row in TMEM only when the warp's row
//     maxima moved.
// Every wait on an mbarrier has an iteration limit; on expiry the kernel sets
// an error bit, skips the rest of its work and still releases its TMEM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "swa_internal.h"

namespace swa {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;        // Q tile rows (M)
constexpr int kKeys = 128;        // keys per KV tile (N of QK^T, K of PV)
constexpr int kThreads = 128;
constexpr int kTileBytes = kRows * kD * 2;   // one 128 x 128 bf16 tile: 32 KB
constexpr int kHalf = kTileBytes / 2;        // one 64-column block: 16 KB
constexpr uint32_t kTmemCols = 256;
constexpr long kSpinLimit = 1L << 26;        // mbarrier polls before giving up

struct TcParams {
  int kind, window, hkv, G, ps, ps_shift;
  KvAddr addr;
  int64_t pool_rows;
  const int32_t *rt;
  int64_t rt_stride;
  const int64_t *req_idx;
  const int64_t *pre;
  const int64_t *seq;
  const int64_t *qo_indptr;
  int bs;
  int qtiles_upper;     // grid.x
  PlanView plan;
  const __nv_bfloat16 *q;
  const float *sinks;
  float scale_log2;
  __nv_bfloat16 *out;
  int max_pages;        // capacity of the per-CTA page-row table
  int32_t *err;
};

// ---------------------------------------------------------------- PTX ---
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
  int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

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
// Waits for the phase with the given parity; false when the poll limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (long i = 0; i < kSpinLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 at [0,14), leading
// byte offset >> 4 at [16,30), stride byte offset >> 4 at [32,46), version 1
// at [46,48), layout (2 = 128-byte swizzle) at [61,64).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), A K-major (bit 15 = 0), B major at bit 16, N >> 3 at
// [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
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
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Byte offset of (row r, 16-byte chunk c in 0..15) inside a 128 x 128 bf16 tile
// stored as two 64-column blocks of [128 rows][128 B] with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ int64_t key_lo(int kind, int window, int64_t p) {
  if (kind == SWA_LAYER_FULL) return 0;
  if (kind == SWA_LAYER_SLIDING) return p - window > 0 ? p - window : 0;
  return (p / window) * window;
}

// Shared memory: [Q 32K][K0 32K][V0 32K][K1 32K][V1 32K][P 32K][page rows][bars]
constexpr int kOffQ = 0;
constexpr int kOffKV = kTileBytes;
constexpr int kOffP = kOffKV + 4 * kTileBytes;
constexpr int kOffRows = kOffP + kTileBytes;

__global__ void __launch_bounds__(kThreads, 1) k_extend_tc(TcParams P) {
  extern __shared__ char smem_raw[];
  // 1024-byte alignment for the swizzled tiles.
  char *smem = reinterpret_cast<char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  int64_t *s_rows = reinterpret_cast<int64_t *>(smem + kOffRows);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffRows + P.max_pages * 8);
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_q0, s_q1, s_pre, s_req;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int kvh = blockIdx.y;
  const int G = P.G;
  const int T = kRows / G;                       // query tokens per tile

  // ---- which Q tile: longest (latest) tiles first ----
  if (tid == 0) {
    int64_t tau = (int64_t)P.qtiles_upper - 1 - blockIdx.x;
    int64_t acc = 0;
    s_req = -1;
    for (int b = 0; b < P.bs; ++b) {
      const int64_t ext = P.qo_indptr[b + 1] - P.qo_indptr[b];
      const int64_t nt = (ext + T - 1) / T;
      if (tau < acc + nt) {
        const int64_t local = (tau - acc) * T;
        s_req = b;
        s_q0 = P.qo_indptr[b] + local;
        s_q1 = min(P.qo_indptr[b + 1], s_q0 + T);
        s_pre = P.pre[b] + local;                 // position of the tile's first query
        break;
      }
      acc += nt;
    }
    s_abort = 0;
  }
  __syncthreads();
  if (s_req < 0) return;
  const int b = (int)s_req;
  const int64_t q0 = s_q0, nq = s_q1 - s_q0, p_first = s_pre;
  const int64_t p_last = p_first + nq - 1;

  // Row of this thread: token tr, head g.
  const int r = tid;
  const int tr = r / G, g = r % G;
  const bool row_valid = tr < nq;
  const int64_t p_row = p_first + tr;
  const int64_t lo_row = key_lo(P.kind, P.window, p_row);

  // Key range of the tile.
  const int64_t k_lo = key_lo(P.kind, P.window, p_first);
  const int64_t k_hi = p_last;
  const int n_tiles = (int)((k_hi - k_lo + kKeys) / kKeys);
  if (k_hi / P.ps - k_lo / P.ps + 1 > P.max_pages) {   // max_seq_len was too small
    if (tid == 0) set_error(P.err, SWA_DEVERR_RANGE);
    return;
  }

  // ---- TMEM ----
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  // ---- page rows of the key range ----
  const int64_t pg0 = k_lo / P.ps;
  const int n_pg = (int)(k_hi / P.ps - pg0 + 1);
  const int64_t page_stride = (int64_t)P.ps * (P.addr.blocks ? P.addr.blocks : 1);
  const int64_t max_page = P.pool_rows / P.ps - 1;
  for (int i = tid; i < n_pg; i += kThreads) {
    const int64_t pos = (pg0 + i) * P.ps > k_lo ? (pg0 + i) * P.ps : k_lo;
    int64_t page;
    if (P.kind == SWA_LAYER_FULL) {
      page = P.rt[P.req_idx[b] * P.rt_stride + pos] / P.ps;
    } else {
      const int32_t *h = P.plan.hdr + b * 4;
      const int64_t k = pos / P.ps - h[2];
      page = (pos >= h[0] && k >= 0 && k < h[3]) ? P.plan.pages[(int64_t)b * P.plan.max_pages + k] : -1;
      if (page == 0) set_error(P.err, SWA_DEVERR_WINDOW_EVICTED);
    }
    if (page < 0 || page > max_page) {
      set_error(P.err, SWA_DEVERR_RANGE);
      page = 0;
    }
    s_rows[i] = page * page_stride;
  }
  // ---- Q tile ----
  const int Hq = P.hkv * G;
  for (int i = tid; i < kRows * 16; i += kThreads) {
    const int rr = i >> 4, c = i & 15;
    const int t2 = rr / G, g2 = rr % G;
    const bool ok = t2 < nq;
    const __nv_bfloat16 *src = P.q + ((q0 + (ok ? t2 : 0)) * Hq + kvh * G + g2) * kD + c * 8;
    cp_async16(sbase + kOffQ + tile_off(rr, c), src, ok);
  }
  __syncthreads();   // page rows, barriers, TMEM address visible
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tS = tmem, tO = tmem + 128;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  const char *kb = P.addr.k + (int64_t)kvh * kD * 2;
  const char *vb = P.addr.v + (int64_t)kvh * kD * 2;
  auto load_kv = [&](int t) {
    const uint32_t dk = sbase + kOffKV + (t & 1) * 2 * kTileBytes;
    const uint32_t dv = dk + kTileBytes;
    const int64_t j0 = k_lo + (int64_t)t * kKeys;
    for (int i = tid; i < kKeys * 16; i += kThreads) {
      const int rr = i >> 4, c = i & 15;
      const int64_t j = j0 + rr;
      const bool ok = j <= k_hi;
      int64_t off = 0;
      if (ok) {
        int64_t pg, in;
        if (P.ps_shift >= 0) {
          pg = j >> P.ps_shift;
          in = j & ((1 << P.ps_shift) - 1);
        } else {
          pg = j / P.ps;
          in = j % P.ps;
        }
        off = (s_rows[pg - pg0] + in) * P.addr.row_bytes + c * 16;
      }
      cp_async16(dk + tile_off(rr, c), kb + off, ok);
      cp_async16(dv + tile_off(rr, c), vb + off, ok);
    }
  };

  load_kv(0);
  cp_commit();

  constexpr uint32_t kIdS = idesc_f16(128, 128, false);
  constexpr uint32_t kIdO = idesc_f16(128, 128, true);
  float m_run = -INFINITY, l_run = 0.f;
  uint32_t phase_s = 0, phase_o = 0;
  bool o_init = false;

  for (int t = 0; t < n_tiles; ++t) {
    if (t + 1 < n_tiles) load_kv(t + 1);
    cp_commit();
    cp_wait<1>();
    fence_async_smem();
    __syncthreads();
    if (s_abort) break;
    const uint32_t kt = sbase + kOffKV + (t & 1) * 2 * kTileBytes;
    const uint32_t vt = kt + kTileBytes;
    // ---- S = Q K^T ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint32_t koff = (ks >> 2) * kHalf + (ks & 3) * 32;
        tc_mma(tS, smem_desc(sbase + kOffQ + koff, 16, 1024), smem_desc(kt + koff, 16, 1024), kIdS,
               ks > 0);
      }
      tc_commit(smem_u32(&bars[0]));
    }
    if (!mbar_wait(smem_u32(&bars[0]), phase_s)) {
      set_error(P.err, SWA_DEVERR_RANGE);
      s_abort = 1;
    }
    phase_s ^= 1;
    tc_fence_after();
    // ---- softmax on this thread's row ----
    const int64_t j0 = k_lo + (int64_t)t * kKeys;
    float s[kKeys];
#pragma unroll
    for (int cb = 0; cb < kKeys / 32; ++cb) {
      uint32_t rr[32];
      TC_LD32(tS + lane_base + cb * 32, rr);
      tc_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) s[cb * 32 + e] = __uint_as_float(rr[e]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < kKeys; ++e) {
      const int64_t j = j0 + e;
      float v = s[e] * P.scale_log2;
      if (!row_valid || j < lo_row || j > p_row) v = -INFINITY;
      s[e] = v;
      mx = fmaxf(mx, v);
    }
    const float m_new = fmaxf(m_run, mx);
    const float mu = m_new == -INFINITY ? 0.f : m_new;
    const float corr = exp2f(m_run - mu);
    float psum = 0.f;
    char *prow = smem + kOffP;
#pragma unroll
    for (int c = 0; c < kKeys / 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a0 = exp2f(s[c * 8 + 2 * e] - mu);
        const float a1 = exp2f(s[c * 8 + 2 * e + 1] - mu);
        __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
        psum += __low2float(h) + __high2float(h);
        w[e] = *reinterpret_cast<uint32_t *>(&h);
      }
      *reinterpret_cast<uint4 *>(prow + tile_off(r, c)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    l_run = l_run * corr + psum;
    m_run = m_new;
    // Rescale this warp's O rows unless no row maximum moved.
    if (o_init && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
      for (int cb = 0; cb < kD / 32; ++cb) {
        uint32_t rr[32];
        TC_LD32(tO + lane_base + cb * 32, rr);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * corr);
        TC_ST32(tO + lane_base + cb * 32, rr);
      }
      tc_wait_st();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- O += P V ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks) {
        const uint32_t aoff = (ks >> 2) * kHalf + (ks & 3) * 32;
        // V as an MN-major operand: 16 keys = 2 swizzle atoms of 8 rows (1024 B
        // apart); the two 64-column blocks of D are 16 KB apart.
        tc_mma(tO, smem_desc(sbase + kOffP + aoff, 16, 1024),
               smem_desc(vt + ks * 16 * 128, kHalf, 1024), kIdO, (o_init || ks > 0) ? 1u : 0u);
      }
      tc_commit(smem_u32(&bars[1]));
    }
    if (!mbar_wait(smem_u32(&bars[1]), phase_o)) {
      set_error(P.err, SWA_DEVERR_RANGE);
      s_abort = 1;
    }
    phase_o ^= 1;
    tc_fence_after();
    o_init = true;
  }
  cp_wait<0>();
  __syncthreads();

  // ---- epilogue: O / (l + sink) ----
  if (!s_abort && o_init) {
    float sg2 = -INFINITY;
    if (P.sinks) sg2 = P.sinks[kvh * G + g] * 1.4426950408889634f;
    const float mfin = fmaxf(m_run == -INFINITY ? 0.f : m_run, sg2);
    const float rsc = exp2f((m_run == -INFINITY ? 0.f : m_run) - mfin);
    const float denom = l_run * rsc + (P.sinks ? exp2f(sg2 - mfin) : 0.f);
    const float f = denom > 0.f ? rsc / denom : 0.f;
    __nv_bfloat16 *orow = P.out + ((q0 + (row_valid ? tr : 0)) * Hq + kvh * G + g) * kD;
#pragma unroll
    for (int cb = 0; cb < kD / 32; ++cb) {
      uint32_t rr[32];
      TC_LD32(tO + lane_base + cb * 32, rr);
      tc_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(rr[e + 2 * k]) * f,
                                                     __uint_as_float(rr[e + 2 * k + 1]) * f);
            w[k] = *reinterpret_cast<uint32_t *>(&h);
          }
          *reinterpret_cast<uint4 *>(orow + cb * 32 + e) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

int tc_max_pages(const Ctx &c, int max_seq_len) {
  return max_seq_len / c.cfg.page_size + 3;
}

}  // namespace

bool tc_extend_supported(const Ctx &c, int layer) {
  if (c.cfg.kv_dtype != SWA_DTYPE_BF16 || c.cfg.head_dim != kD) return false;
  if (c.cfg.page_size < 16) return false;
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
  P.ps_shift = (P.ps & (P.ps - 1)) == 0 ? __builtin_ctz((unsigned)P.ps) : -1;
  P.addr = L.addr;
  P.pool_rows = (L.in_full ? c.cfg.size_full : c.cfg.size_swa) + c.cfg.page_size;
  P.rt = a.rt;
  P.rt_stride = a.rt_stride;
  P.req_idx = a.req_idx;
  P.pre = a.pre;
  P.seq = a.seq;
  P.qo_indptr = a.qo_indptr;
  P.bs = a.bs;
  const int T = kRows / P.G;
  P.qtiles_upper = (int)((a.nq + T - 1) / T + a.bs);
  P.plan = a.plan;
  P.q = static_cast<const __nv_bfloat16 *>(a.q);
  P.sinks = a.sinks;
  P.scale_log2 = a.scale * 1.4426950408889634f;
  P.out = static_cast<__nv_bfloat16 *>(a.out);
  P.max_pages = tc_max_pages(c, a.max_seq_len);
  P.err = c.err_word;
  const size_t smem = 1024 + kOffRows + (size_t)P.max_pages * 8 + 64;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_extend_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(P.qtiles_upper, L.hkv);
  k_extend_tc<<<grid, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace swa
