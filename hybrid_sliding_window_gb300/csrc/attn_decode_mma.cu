// Tensor-core paged decode attention for bf16 and FP8-E4M3 KV (D = 64 / 128,
// GQA group G <= 16).
//
// Method: "SWA in SGLang" design note - sliding layers read the window of
// Wx+1 keys through the per-batch SWA page table, full layers every key
// through req_to_token; a per-head sink logit joins the denominator.
//
// GB300 design.  Decode is bound by HBM: each key costs 4*D*G flops per KV
// head on 2*D*b bytes, i.e. 2G/b flop/byte (16 for MiMo's full layers), which
// CUDA-core FMAs cannot sustain at HBM speed, so the QK^T and PV products run
// on tensor cores with the G query heads of one KV head as the M=16 rows of
// mma.m16n8k16 (unused rows are zero).  Work item = (request, KV head, split
// of 1024 to 4096 keys, a power of two chosen per launch from the longest
// request); a CTA of 4 warps streams 64-key tiles through a
// 3-stage cp.async pipeline (16-byte gathers of whole K/V rows, row address
// from the index tables, out-of-range rows zero-filled without a read), each
// warp owning 16 keys of every tile with its own online-softmax state in
// registers.  FP8 rows are converted to f16 in registers on their way to
// the tensor cores (E4M3 is a subset
// of f16; the scales fold into the score scale and the output).  Splits of
// one (request, KV head) meet through an atomic ticket: the last CTA merges
// the partials and the sink, so one launch does split and merge.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kv_codec.cuh"
#include "split_merge.cuh"
#include "swa_internal.h"

namespace swa {
namespace {


struct MmaParams {
  int kind, window, hkv, G, ps;
  int ps_shift;          // log2(ps) when ps is a power of two, else -1
  KvAddr addr;
  int64_t pool_rows;
  const int32_t *rt;
  int64_t rt_stride;
  const int64_t *req_idx;
  const int64_t *seq;
  PlanView plan;
  const __nv_bfloat16 *q;
  const float *sinks;
  float qk_scale_log2;   // sm_scale * log2(e) * k_scale
  float v_scale;
  __nv_bfloat16 *out;
  float *partials;
  int32_t *tickets;
  int max_splits;
  int split_keys;         // keys per split (a multiple of the tile)
  int32_t *err;
  // Optional store of the new tokens ([bs][hkv][D] bf16 rows) before reading:
  // the slot is full_loc (full layers), else swa_loc, else mapping[full_loc].
  const char *k_new, *v_new;
  const int64_t *full_loc, *swa_loc, *mapping;
  int64_t map_len;
  int in_full;
  float st_k_scale, st_v_scale;
};

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

// The SFU's base-2 exponential (denormal results flush to zero: weights below
// 2^-126 of the row maximum).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
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

// Per-request table entry points, read once at the start of a CTA (they do
// not depend on the sequence length, so their loads overlap with it): the
// req_to_token row of a full layer, the plan header of a windowed one.
struct ReqRef {
  int64_t row;           // full: req_idx[b]
  int32_t h0, h2, h3;    // windowed: first planned position, first page, page count
};

__device__ __forceinline__ ReqRef req_ref(const MmaParams &P, int b) {
  ReqRef r{0, 0, 0, 0};
  if (P.kind == SWA_LAYER_FULL) {
    r.row = P.req_idx[b];
  } else {
    const int32_t *h = P.plan.hdr + b * 4;
    r.h0 = h[0];
    r.h2 = h[2];
    r.h3 = h[3];
  }
  return r;
}

__device__ __forceinline__ int64_t key_slot(const MmaParams &P, const ReqRef &R, int b, int64_t j) {
  if (P.kind == SWA_LAYER_FULL) return P.rt[R.row * P.rt_stride + j];
  const int64_t k = j / P.ps - R.h2;
  if (j < R.h0 || k < 0 || k >= R.h3) {
    set_error(P.err, SWA_DEVERR_RANGE);
    return 0;
  }
  const int64_t page = P.plan.pages[(int64_t)b * P.plan.max_pages + k];
  if (page <= 0) set_error(P.err, SWA_DEVERR_WINDOW_EVICTED);
  return page * P.ps + j % P.ps;
}

// The new token's row of KV head kvh for request b, written to the pool by
// the CTA whose key range ends at that token (the only one that reads it);
// the same bytes as the KV store kernel writes.
template <int D, bool FP8>
__device__ __forceinline__ void store_new_token(const MmaParams &P, int b, int kvh, int tid,
                                                int nthreads) {
  constexpr int kEsz = FP8 ? 1 : 2;
  constexpr int kChunks = D * kEsz / 16;   // 16-byte pool chunks of one head row
  int64_t slot;
  if (P.in_full) {
    slot = P.full_loc[b];
  } else if (P.swa_loc) {
    slot = P.swa_loc[b];
  } else {
    int64_t f = P.full_loc[b];
    if (f < 0) f += P.map_len;
    slot = (f >= 0 && f < P.map_len) ? P.mapping[f] : -1;
  }
  if (slot < 0 || slot >= P.pool_rows) {
    if (tid == 0) set_error(P.err, SWA_DEVERR_RANGE);
    return;
  }
  const int64_t row = kv_row(P.addr, slot) * P.addr.row_bytes + (int64_t)kvh * D * kEsz;
  const int64_t src_row = ((int64_t)b * P.hkv + kvh) * D * 2;   // bf16 input
  for (int i = tid; i < 2 * kChunks; i += nthreads) {
    const bool is_v = i >= kChunks;
    const int c = is_v ? i - kChunks : i;
    char *dst = (is_v ? P.addr.v : P.addr.k) + row + c * 16;
    const char *src = (is_v ? P.v_new : P.k_new) + src_row;
    if constexpr (FP8) {
      const uint4 *w = reinterpret_cast<const uint4 *>(src + c * 32);
      *reinterpret_cast<uint4 *>(dst) = e4m3_encode16(w[0], w[1], is_v ? P.st_v_scale : P.st_k_scale);
    } else {
      *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src + c * 16);
    }
  }
}

// Shared-memory plan (bytes):
//   Q tile      16 x D  16-bit, swizzled                      : 32*D
//   stages      kStages x (K,V) 64 x D stored elements         : kStages*2*64*D*esz
// Heads-as-rows (G > 8) FP8 stages are half the size of bf16 ones, so twice
// as many fit at 2 CTAs per SM; keys-as-rows kernels need fewer registers and
// run 4 CTAs per SM where the tiles allow.
template <int D, bool FP8, bool KM, int NW>
struct Smem {
  static constexpr int kWarps = NW;
  static constexpr int kTile = 16 * NW;   // keys per stage: 16 per warp
  static constexpr int kEsz = FP8 ? 1 : 2;
  static constexpr int kStages = (FP8 && !KM) ? 6 : 3;
  static constexpr int kQ = 16 * D * 2;
  static constexpr int kStageBytes = 2 * kTile * D * kEsz;
  // warp rows of O (D + 4 floats each), then per-row max, sum and weight
  static constexpr int kMerge = kWarps * 16 * (D + 4) * 4 + 3 * kWarps * 16 * 4;
  static constexpr int kMain = kQ + kStages * kStageBytes;
  static constexpr int kBig = kMain > kMerge ? kMain : kMerge;
  static constexpr int kTotal = kBig > kMergeScratchBytes ? kBig : kMergeScratchBytes;
  static constexpr int kMinBlocks =
      NW == 2 ? (D == 64 ? 8 : 4) : ((D == 64 || (KM && FP8)) ? 4 : 2);
};

// 16-bit tile addressing: row r, 16-byte chunk c (D/8 chunks per row), XOR swizzle.
template <int D>
__device__ __forceinline__ int swz(int r, int c) {
  return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

// FP8 tiles: row r of D bytes, 16-byte chunk c.  K rows are read by ldmatrix
// (eight rows, one chunk), V rows as 32-bit words by lanes that own key pairs
// (2c4, 2c4+1): each tile has the swizzle that keeps its reads free of bank
// conflicts (for D = 128; D = 64 V reads are two-way).
template <int D>
__device__ __forceinline__ int kswz8(int r, int c) {
  return r * D + ((c ^ (D == 128 ? (r & 7) : ((r >> 1) & 3))) << 4);
}
template <int D>
__device__ __forceinline__ int vswz8(int r, int c) {
  return r * D + ((c ^ (D == 128 ? 2 * ((r >> 1) & 3) : 2 * ((r >> 1) & 1))) << 4);
}

// Four E4M3 values (bytes 0..3 of w) to two f16 pairs, (b0, b1) and (b2, b3),
// low byte in the low half; exact (E4M3 is a subset of f16).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Transpose of an 8x8 16-bit block held one row-pair per lane.
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

struct CtaSync {
  __device__ void operator()() const { __syncthreads(); }
};

// Two orientations of the per-warp products (16 keys of each 64-key tile per
// warp):
//  * heads as rows (KM = false, G <= 16): S = Q K^T with the G heads as the
//    M = 16 rows, then O += P V;
//  * keys as rows (KM = true, G <= 8): S^T = K Q^T with the 16 keys as M and
//    the heads as N = 8, then O^T += V^T P^T, P^T transposed in registers.
//    Half the tensor-core work when the group has at most 8 heads, and half
//    the accumulator registers.
template <int D, bool FP8, bool KM, int NW>
__global__ void __launch_bounds__(NW * 32, (Smem<D, FP8, KM, NW>::kMinBlocks))
    k_decode_mma(MmaParams P) {
  using S = Smem<D, FP8, KM, NW>;
  constexpr int kWarps = NW;
  constexpr int kTile = S::kTile;
  static_assert(S::kTotal >= kMergeScratchBytes, "merge scratch exceeds the tiles");
  constexpr bool F16 = FP8;                 // FP8 KV widens to f16; bf16 KV stays bf16
  constexpr int kStages = S::kStages;
  constexpr int kEsz = S::kEsz;
  constexpr int kRowChunks = D * kEsz / 16; // 16-byte chunks of one stored head row
  extern __shared__ __align__(128) char smem[];
  char *sq = smem;
  char *sstage = smem + S::kQ;

  // KV heads fastest: the CTAs of all heads of the same keys run together, so
  // each token's interleaved head rows are read from DRAM at about one time.
  // Split index slowest: every request's leading (full-length) splits are
  // dispatched first and the last wave holds the ragged final splits of the
  // longest requests, which shortens the tail.
  const int kvh = blockIdx.x, b = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G;
  const int Hq = P.hkv * G;

  // Launched as a programmatic dependent of the previous kernel on the
  // stream.  The index tables read first (sequence length, plan, req_to_token)
  // come from the allocation and plan kernels, which completed before the
  // previous kernel passed its own wait, so they are read before this
  // kernel's wait and their latency overlaps the previous kernel's tail;
  // everything the previous kernel may write (q, the new token's K/V, the
  // workspace) and the tile loads come after the wait.
  const ReqRef R = req_ref(P, b);
  // Windowed layers whose plan row fits one warp: the row's page entries are
  // read now, with the sequence length and the plan header, instead of after
  // them (one dependent DRAM round trip fewer before the first tile).
  const bool pfast = P.kind != SWA_LAYER_FULL && P.plan.max_pages <= 32;
  int32_t pv = 0;
  if (pfast && warp == 0 && lane < P.plan.max_pages)
    pv = P.plan.pages[(int64_t)b * P.plan.max_pages + lane];
  const int64_t p = P.seq[b] - 1;
  int64_t lo = 0;
  if (P.kind == SWA_LAYER_SLIDING) lo = p - P.window > 0 ? p - P.window : 0;
  else if (P.kind == SWA_LAYER_CHUNKED) lo = (p / P.window) * P.window;
  const int64_t n_keys = p - lo + 1;
  const int n_splits = (int)((n_keys + P.split_keys - 1) / P.split_keys);
  if (split >= n_splits) return;
  const int64_t k0 = lo + (int64_t)split * P.split_keys;
  const int64_t k1 = min(p + 1, k0 + P.split_keys);
  const int n_tiles = (int)((k1 - k0 + kTile - 1) / kTile);

  // ---- pages of this split, looked up once (one table read per page) ----
  // Positions of one page occupy consecutive slots of one pool page, so key j
  // sits (j % ps) rows past the first row of page j / ps; the table holds the
  // byte offset of that first row.
  int64_t *s_rb = reinterpret_cast<int64_t *>(smem + S::kTotal);
  const int rb = (int)P.addr.row_bytes;
  const int64_t pg0 = k0 / P.ps;
  const int n_pg = (int)((k1 - 1) / P.ps - pg0 + 1);
  const int64_t page_stride = (int64_t)P.ps * (P.addr.blocks ? P.addr.blocks : 1);
  const int64_t max_page = (P.pool_rows / P.ps) - 1;
  if (pfast) {
    // n_pg <= plan pages <= 32: warp 0, lane i takes page pg0 + i from the
    // lane that read its plan entry (the same checks as key_slot).
    if (warp == 0) {
      const int64_t pos = (pg0 + lane) * P.ps > k0 ? (pg0 + lane) * P.ps : k0;
      const int64_t k = pos / P.ps - R.h2;
      const int32_t pgv = __shfl_sync(0xffffffffu, pv, (int)(k < 0 ? 0 : (k > 31 ? 31 : k)));
      if (lane < n_pg) {
        int64_t slot = 0;
        if (pos < R.h0 || k < 0 || k >= R.h3) {
          set_error(P.err, SWA_DEVERR_RANGE);
        } else {
          if (pgv <= 0) set_error(P.err, SWA_DEVERR_WINDOW_EVICTED);
          slot = (int64_t)pgv * P.ps + pos % P.ps;
        }
        int64_t page = slot / P.ps;
        if (slot < 0 || page > max_page) {
          set_error(P.err, SWA_DEVERR_RANGE);
          page = 0;
        }
        s_rb[lane] = page * page_stride * rb;
      }
    }
  }
  for (int i = pfast ? n_pg : tid; i < n_pg; i += blockDim.x) {
    const int64_t pos = (pg0 + i) * P.ps > k0 ? (pg0 + i) * P.ps : k0;
    const int64_t slot = key_slot(P, R, b, pos);
    int64_t page = slot / P.ps;
    if (slot < 0 || page > max_page) {
      set_error(P.err, SWA_DEVERR_RANGE);
      page = 0;
    }
    s_rb[i] = page * page_stride * rb;
  }

  // The previous kernel's memory is needed from here on.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // The next kernel on the stream may launch once every CTA of this grid has
  // got here (all of them are resident by then): its CTAs read their own
  // index tables while this grid streams, and wait for it to complete before
  // touching anything it writes.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  // ---- Q rows into registers: their latency hides behind the first tile
  // loads ----
  constexpr int kQPer = 16 * (D / 8) / (kWarps * 32);
  uint4 qv[kQPer];
#pragma unroll
  for (int k = 0; k < kQPer; ++k) {
    const int i = tid + k * kWarps * 32;
    const int r = i / (D / 8), c = i % (D / 8);
    qv[k] = make_uint4(0, 0, 0, 0);
    if (r < G) qv[k] = *reinterpret_cast<const uint4 *>(P.q + ((int64_t)b * Hq + kvh * G + r) * D + c * 8);
  }

  // ---- tile loader ----
  const char *kbase = P.addr.k + (int64_t)kvh * D * kEsz;
  const char *vbase = P.addr.v + (int64_t)kvh * D * kEsz;
  const int ps_shift = P.ps_shift;
  // Each thread copies one fixed 16-byte chunk c of rows r0, r0 + kRowStep,
  // ... of every tile (K and V), so its global and shared addresses change
  // only by the row; positions are counted from the first row of page pg0.
  constexpr int kThreads = kWarps * 32;
  constexpr int kRowStep = kThreads / kRowChunks;
  constexpr int kPasses = kTile / kRowStep;
  static_assert(kTile % kRowStep == 0, "whole passes per tile");
  const int lc = tid % kRowChunks, lr0 = tid / kRowChunks;
  const char *kb_c = kbase + lc * 16, *vb_c = vbase + lc * 16;
  const int o0 = (int)(k0 - pg0 * P.ps);
  const int pmask = ps_shift >= 0 ? (1 << ps_shift) - 1 : 0;
  auto load_tile = [&](int t) {
    char *st = sstage + (t % kStages) * S::kStageBytes;
    const int x0 = o0 + t * kTile;
    const int nv = (int)min((int64_t)kTile, k1 - (k0 + (int64_t)t * kTile));
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
      const int r = lr0 + k * kRowStep;
      const bool ok = r < nv;
      const int x = x0 + r;
      int pi, in;
      if (ps_shift >= 0) {
        pi = x >> ps_shift;
        in = x & pmask;
      } else {
        pi = x / P.ps;
        in = x - pi * P.ps;
      }
      const int64_t off = ok ? s_rb[pi] + (int64_t)in * rb : 0;
      int dk, dv;
      if constexpr (FP8) {
        dk = kswz8<D>(r, lc);
        dv = kTile * D + vswz8<D>(r, lc);
      } else {
        dk = swz<D>(r, lc);
        dv = kTile * D * 2 + dk;
      }
      cp_async16(smem_u32(st + dk), kb_c + off, ok);
      cp_async16(smem_u32(st + dv), vb_c + off, ok);
    }
  };
  // The new token (fused store): written before the barrier below, so the
  // tile loads issued after it read the stored row.
  if (P.k_new != nullptr && k1 == p + 1) store_new_token<D, FP8>(P, b, kvh, tid, kThreads);
  __syncthreads();  // page rows (and the new token's row) visible
#pragma unroll
  for (int t = 0; t < kStages - 1; ++t) {
    if (t < n_tiles) load_tile(t);
    cp_commit();
  }

  // ---- Q tile (rows >= G zero), f16 for FP8 KV ----
#pragma unroll
  for (int k = 0; k < kQPer; ++k) {
    const int i = tid + k * kWarps * 32;
    const int r = i / (D / 8), c = i % (D / 8);
    uint4 v = qv[k];
    if constexpr (F16) {
      const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&v);
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) w[e] = pack2<true>(__bfloat162float(h[2 * e]), __bfloat162float(h[2 * e + 1]));
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4 *>(sq + swz<D>(r, c)) = v;
  }
  __syncthreads();  // Q tile visible

  const int g = lane >> 2, c4 = lane & 3;
  // Q fragments.  FP8: the K fragments of a 16-dim step carry dims 4c4, 4c4+1
  // at k = 2c4, 2c4+1 and dims 4c4+2, 4c4+3 at k = 2c4+8, 2c4+9 (one 32-bit
  // word of E4M3 per key row), so Q takes the same order of dims.
  constexpr int kQF = KM ? 2 : 4;
  uint32_t qa[D / 16][kQF];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    if constexpr (KM) {   // B = Q^T: head g, two dim pairs
      const char *r0 = FP8 ? sq + swz<D>(g, 2 * ks + (c4 >> 1)) + (c4 & 1) * 8
                           : sq + swz<D>(g, 2 * ks) + 4 * c4;
      qa[ks][0] = *reinterpret_cast<const uint32_t *>(r0);
      qa[ks][1] = FP8 ? *reinterpret_cast<const uint32_t *>(r0 + 4)
                      : *reinterpret_cast<const uint32_t *>(sq + swz<D>(g, 2 * ks + 1) + 4 * c4);
    } else if constexpr (FP8) {
      const int off = (c4 & 1) * 8;
      const char *r0 = sq + swz<D>(g, 2 * ks + (c4 >> 1)) + off;
      const char *r1 = sq + swz<D>(g + 8, 2 * ks + (c4 >> 1)) + off;
      qa[ks][0] = *reinterpret_cast<const uint32_t *>(r0);
      qa[ks][1] = *reinterpret_cast<const uint32_t *>(r1);
      qa[ks][2] = *reinterpret_cast<const uint32_t *>(r0 + 4);
      qa[ks][3] = *reinterpret_cast<const uint32_t *>(r1 + 4);
    } else {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = ks * 2 + (lane >> 4);
      uint32_t *f = qa[ks];
      ldsm_x4(smem_u32(sq + swz<D>(r, c)), f[0], f[1], f[2], f[3]);
    }
  }

  // Accumulators.  Heads as rows: o[n] = O[heads g, g+8][dims of block n];
  // m0/l0 row g, m1/l1 row g+8.  Keys as rows: o[mt] = O^T[dims of block mt]
  // [heads 2c4, 2c4+1]; m0/l0 head 2c4, m1/l1 head 2c4+1 (l per lane until
  // the end).
  constexpr int kOB = KM ? D / 16 : D / 8;
  float o[kOB][4];
#pragma unroll
  for (int n = 0; n < kOB; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int t = 0; t < n_tiles; ++t) {
    cp_wait<kStages - 2>();
    __syncthreads();
    if (t + kStages - 1 < n_tiles) load_tile(t + kStages - 1);
    cp_commit();
    const char *st = sstage + (t % kStages) * S::kStageBytes;
    const char *tv = st + kTile * D * kEsz;
    // keys of this tile at or past nvt are outside the split (last tile only)
    const int nvt = (int)min((int64_t)kTile, k1 - (k0 + (int64_t)t * kTile));
    const int jw = warp * 16;
    if constexpr (KM) {
      // ---- S^T = K Q^T: rows = this warp's 16 keys, columns = heads ----
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      const int kr = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
      if constexpr (FP8) {
#pragma unroll
        for (int kp = 0; kp < D / 32; ++kp) {   // two 16-dim steps per ldmatrix
          uint32_t w[4];
          ldsm_x4(smem_u32(st + kswz8<D>(kr, 2 * kp + (lane >> 4))), w[0], w[1], w[2], w[3]);
          uint32_t a0[4], a1[4];
          e4m3x4_to_f16x2x2(w[0], a0[0], a0[2]);
          e4m3x4_to_f16x2x2(w[1], a0[1], a0[3]);
          e4m3x4_to_f16x2x2(w[2], a1[0], a1[2]);
          e4m3x4_to_f16x2x2(w[3], a1[1], a1[3]);
          mma16816<true>(sa, a0, qa[2 * kp][0], qa[2 * kp][1]);
          mma16816<true>(sb, a1, qa[2 * kp + 1][0], qa[2 * kp + 1][1]);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t a[4];
          ldsm_x4(smem_u32(st + swz<D>(kr, 2 * ks + (lane >> 4))), a[0], a[1], a[2], a[3]);
          mma16816<false>((ks & 1) ? sb : sa, a, qa[ks][0], qa[ks][1]);
        }
      }
      // sa: (key g, head 2c4), (key g, head 2c4+1), (key g+8, head 2c4), (key g+8, head 2c4+1)
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = (sa[e] + sb[e]) * P.qk_scale_log2;
      if (nvt < kTile) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (jw + g + (e >> 1) * 8 >= nvt) v[e] = -INFINITY;
      }
      float r0 = fmaxf(v[0], v[2]), r1 = fmaxf(v[1], v[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        r0 = fmaxf(r0, __shfl_xor_sync(0xffffffffu, r0, off));
        r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, off));
      }
      const float mn0 = fmaxf(m0, r0), mn1 = fmaxf(m1, r1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float corr0 = ex2(m0 - mu0), corr1 = ex2(m1 - mu1);
      m0 = mn0;
      m1 = mn1;
      v[0] = ex2(v[0] - mu0);
      v[2] = ex2(v[2] - mu0);
      v[1] = ex2(v[1] - mu1);
      v[3] = ex2(v[3] - mu1);
      l0 = l0 * corr0 + (v[0] + v[2]);
      l1 = l1 * corr1 + (v[1] + v[3]);
      if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {
#pragma unroll
        for (int n = 0; n < kOB; ++n) {
          o[n][0] *= corr0;
          o[n][1] *= corr1;
          o[n][2] *= corr0;
          o[n][3] *= corr1;
        }
      }
      // P^T as the B operand: lane (g, c4) wants keys 2c4, 2c4+1 (and +8) of
      // head g, the transpose of what it holds.
      const uint32_t pb0 = movm_t(pack2<F16>(v[0], v[1]));
      const uint32_t pb1 = movm_t(pack2<F16>(v[2], v[3]));
      // ---- O^T += V^T P^T ----
      if constexpr (FP8) {
        // Lane (g, c4) reads one word (dims 4w..4w+3, w = g + 8wg) of key rows
        // 2c4, 2c4+1, 2c4+8, 2c4+9 and pairs the keys byte-wise: block 2wg
        // carries dims 4w (row g) and 4w+1 (row g+8), block 2wg+1 dims 4w+2
        // and 4w+3.  The output is un-permuted when it leaves the registers.
        const int r0v = warp * 16 + 2 * c4;
#pragma unroll
        for (int wg = 0; wg < D / 32; ++wg) {
          const int w = g + 8 * wg, c = w >> 2, wo = (w & 3) * 4;
          const uint32_t x0 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0v, c) + wo);
          const uint32_t y0 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0v + 1, c) + wo);
          const uint32_t x1 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0v + 8, c) + wo);
          const uint32_t y1 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0v + 9, c) + wo);
          const uint32_t lo0 = __byte_perm(x0, y0, 0x5140), hi0 = __byte_perm(x0, y0, 0x7362);
          const uint32_t lo1 = __byte_perm(x1, y1, 0x5140), hi1 = __byte_perm(x1, y1, 0x7362);
          uint32_t a0[4], a1[4];
          e4m3x4_to_f16x2x2(lo0, a0[0], a0[1]);
          e4m3x4_to_f16x2x2(lo1, a0[2], a0[3]);
          e4m3x4_to_f16x2x2(hi0, a1[0], a1[1]);
          e4m3x4_to_f16x2x2(hi1, a1[2], a1[3]);
          mma16816<true>(o[2 * wg], a0, pb0, pb1);
          mma16816<true>(o[2 * wg + 1], a1, pb0, pb1);
        }
      } else {
        const int vr = warp * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          uint32_t a[4];
          ldsm_x4_t(smem_u32(tv + swz<D>(vr, 2 * mt + ((lane >> 3) & 1))), a[0], a[1], a[2], a[3]);
          mma16816<false>(o[mt], a, pb0, pb1);
        }
      }
    } else {
      // ---- S = Q K^T for this warp's 16 keys ----
      // Two accumulators per 8-key block halve the dependent mma chain.
      float s[2][4], sx[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = sx[nt][e] = 0.f;
        const int r = warp * 16 + nt * 8 + (lane & 7);
        if constexpr (FP8) {
          // ldmatrix of raw E4M3 rows: register j holds 4 dims of chunk 4kq+j.
#pragma unroll
          for (int kq = 0; kq < D / 64; ++kq) {
            uint32_t w[4];
            ldsm_x4(smem_u32(st + kswz8<D>(r, kq * 4 + (lane >> 3))), w[0], w[1], w[2], w[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t lo, hi;
              e4m3x4_to_f16x2x2(w[j], lo, hi);
              mma16816<true>((j & 1) ? sx[nt] : s[nt], qa[kq * 4 + j], lo, hi);
            }
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            const int c = kk * 4 + (lane >> 3);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(smem_u32(st + swz<D>(r, c)), b0, b1, b2, b3);
            mma16816<false>(s[nt], qa[2 * kk], b0, b1);
            mma16816<false>(sx[nt], qa[2 * kk + 1], b2, b3);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] += sx[nt][e];
      }
      // Scale, mask, online softmax (rows g and g+8).
      float rmax0 = -INFINITY, rmax1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] *= P.qk_scale_log2;
        if (nvt < kTile) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (jw + nt * 8 + 2 * c4 + (e & 1) >= nvt) s[nt][e] = -INFINITY;
        }
        rmax0 = fmaxf(rmax0, fmaxf(s[nt][0], s[nt][1]));
        rmax1 = fmaxf(rmax1, fmaxf(s[nt][2], s[nt][3]));
      }
      rmax0 = fmaxf(rmax0, __shfl_xor_sync(0xffffffffu, rmax0, 1));
      rmax0 = fmaxf(rmax0, __shfl_xor_sync(0xffffffffu, rmax0, 2));
      rmax1 = fmaxf(rmax1, __shfl_xor_sync(0xffffffffu, rmax1, 1));
      rmax1 = fmaxf(rmax1, __shfl_xor_sync(0xffffffffu, rmax1, 2));
      const float mn0 = fmaxf(m0, rmax0), mn1 = fmaxf(m1, rmax1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float corr0 = ex2(m0 - mu0), corr1 = ex2(m1 - mu1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = ex2(s[nt][0] - mu0);
        s[nt][1] = ex2(s[nt][1] - mu0);
        s[nt][2] = ex2(s[nt][2] - mu1);
        s[nt][3] = ex2(s[nt][3] - mu1);
        ps0 += s[nt][0] + s[nt][1];
        ps1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * corr0 + ps0;
      l1 = l1 * corr1 + ps1;
      if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {   // a row maximum moved
#pragma unroll
        for (int n = 0; n < kOB; ++n) {
          o[n][0] *= corr0;
          o[n][1] *= corr0;
          o[n][2] *= corr1;
          o[n][3] *= corr1;
        }
      }
      uint32_t pa[4];
      pa[0] = pack2<F16>(s[0][0], s[0][1]);
      pa[1] = pack2<F16>(s[0][2], s[0][3]);
      pa[2] = pack2<F16>(s[1][0], s[1][1]);
      pa[3] = pack2<F16>(s[1][2], s[1][3]);
      // ---- O += P V ----
      if constexpr (FP8) {
        // Lane (g, c4) needs V at keys (2c4, 2c4+1) and (2c4+8, 2c4+9) for
        // one output column per 8-column block: it reads one word (4 dims) of
        // each of those four rows and pairs the keys byte-wise, so n-block
        // 4ng+q carries dim 4(n + 8ng) + q at column n.  The output is
        // un-permuted when it leaves the registers.
        const int r0 = warp * 16 + 2 * c4;
#pragma unroll
        for (int ng = 0; ng < D / 32; ++ng) {
          const int w = g + 8 * ng, c = w >> 2, wo = (w & 3) * 4;
          const uint32_t a0 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0, c) + wo);
          const uint32_t b0 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0 + 1, c) + wo);
          const uint32_t a1 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0 + 8, c) + wo);
          const uint32_t b1 = *reinterpret_cast<const uint32_t *>(tv + vswz8<D>(r0 + 9, c) + wo);
          const uint32_t lo0 = __byte_perm(a0, b0, 0x5140), hi0 = __byte_perm(a0, b0, 0x7362);
          const uint32_t lo1 = __byte_perm(a1, b1, 0x5140), hi1 = __byte_perm(a1, b1, 0x7362);
          uint32_t l0a, l0b, l1a, l1b, h0a, h0b, h1a, h1b;
          e4m3x4_to_f16x2x2(lo0, l0a, l0b);
          e4m3x4_to_f16x2x2(lo1, l1a, l1b);
          e4m3x4_to_f16x2x2(hi0, h0a, h0b);
          e4m3x4_to_f16x2x2(hi1, h1a, h1b);
          mma16816<true>(o[4 * ng + 0], pa, l0a, l1a);
          mma16816<true>(o[4 * ng + 1], pa, l0b, l1b);
          mma16816<true>(o[4 * ng + 2], pa, h0a, h1a);
          mma16816<true>(o[4 * ng + 3], pa, h0b, h1b);
        }
      } else {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int c = dp * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(tv + swz<D>(r, c)), b0, b1, b2, b3);
          mma16816<false>(o[2 * dp], pa, b0, b1);
          mma16816<false>(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
  }
  cp_wait<0>();
  if constexpr (KM) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  } else {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  __syncthreads();  // stages no longer needed: reuse for the warp merge

  constexpr int OS = D + 4;
  float *sm_o = reinterpret_cast<float *>(smem);
  float *sm_m = sm_o + kWarps * 16 * OS;
  float *sm_l = sm_m + kWarps * 16;
  if constexpr (KM) {
    if (g == 0) {
      sm_m[warp * 16 + 2 * c4] = m0;
      sm_m[warp * 16 + 2 * c4 + 1] = m1;
      sm_l[warp * 16 + 2 * c4] = l0;
      sm_l[warp * 16 + 2 * c4 + 1] = l1;
    }
    float *h0p = sm_o + (warp * 16 + 2 * c4) * OS;
    float *h1p = h0p + OS;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      // Dims of accumulator rows g and g+8 (FP8: as the V pairing gave them).
      const int da = FP8 ? 4 * (g + 8 * (mt >> 1)) + 2 * (mt & 1) : mt * 16 + g;
      const int db = FP8 ? da + 1 : da + 8;
      h0p[da] = o[mt][0];
      h1p[da] = o[mt][1];
      h0p[db] = o[mt][2];
      h1p[db] = o[mt][3];
    }
  } else {
    if (c4 == 0) {
      sm_m[warp * 16 + g] = m0;
      sm_m[warp * 16 + g + 8] = m1;
      sm_l[warp * 16 + g] = l0;
      sm_l[warp * 16 + g + 8] = l1;
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      // Columns of accumulator block n (FP8: the dims the V pairing gave them).
      const int d0 = FP8 ? 4 * (2 * c4 + 8 * (n >> 2)) + (n & 3) : n * 8 + 2 * c4;
      const int d1 = FP8 ? d0 + 4 : d0 + 1;
      float *r0p = sm_o + (warp * 16 + g) * OS;
      float *r1p = sm_o + (warp * 16 + g + 8) * OS;
      r0p[d0] = o[n][0];
      r0p[d1] = o[n][1];
      r1p[d0] = o[n][2];
      r1p[d1] = o[n][3];
    }
  }
  __syncthreads();

  const bool single = n_splits == 1;
  const int pstride = part_stride(G, D);
  const int64_t pair = (int64_t)b * P.hkv + kvh;
  float *part = P.partials + (pair * P.max_splits + split) * pstride;
  // Row statistics once per head (one thread each): the weight of every
  // warp's partial row, with the softmax denominator and the sink folded in
  // when this split is the whole request.
  float *s_cf = sm_l + kWarps * 16;   // [kWarps][16]
  if (tid < G) {
    const int gg = tid;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 16 + gg]);
    const float Mu = M == -INFINITY ? 0.f : M;
    float f[kWarps], L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      f[w] = exp2f(sm_m[w * 16 + gg] - Mu);
      L += sm_l[w * 16 + gg] * f[w];
    }
    float scale = 1.f;
    if (single) {
      float Mf = Mu, extra = 0.f;
      if (P.sinks) {
        const float sg = P.sinks[kvh * G + gg] * 1.4426950408889634f;
        Mf = fmaxf(Mu, sg);
        extra = exp2f(sg - Mf);
      }
      const float r = exp2f(Mu - Mf);
      scale = r * P.v_scale / (L * r + extra);
    } else {
      part[G * D + 2 * gg] = Mu;
      part[G * D + 2 * gg + 1] = L;
    }
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s_cf[w * 16 + gg] = f[w] * scale;
  }
  __syncthreads();
  // Eight dims per thread and pass: weighted sum of the warps' rows, then one
  // 16-byte bf16 store (whole request) or two float4 partial stores.
  for (int e8 = tid; e8 < G * (D / 8); e8 += kThreads) {
    const int gg = e8 / (D / 8), d0 = (e8 % (D / 8)) * 8;
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float cf = s_cf[w * 16 + gg];
      const float4 x = *reinterpret_cast<const float4 *>(sm_o + (w * 16 + gg) * OS + d0);
      const float4 y = *reinterpret_cast<const float4 *>(sm_o + (w * 16 + gg) * OS + d0 + 4);
      a[0] += cf * x.x; a[1] += cf * x.y; a[2] += cf * x.z; a[3] += cf * x.w;
      a[4] += cf * y.x; a[5] += cf * y.y; a[6] += cf * y.z; a[7] += cf * y.w;
    }
    if (single) {
      uint4 packed;
      packed.x = pack2<false>(a[0], a[1]);
      packed.y = pack2<false>(a[2], a[3]);
      packed.z = pack2<false>(a[4], a[5]);
      packed.w = pack2<false>(a[6], a[7]);
      *reinterpret_cast<uint4 *>(P.out + ((int64_t)b * Hq + kvh * G + gg) * D + d0) = packed;
    } else {
      *reinterpret_cast<float4 *>(part + gg * D + d0) = make_float4(a[0], a[1], a[2], a[3]);
      *reinterpret_cast<float4 *>(part + gg * D + d0 + 4) = make_float4(a[4], a[5], a[6], a[7]);
    }
  }
  if (single) return;
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&P.tickets[pair], 1);
    s_last = prev == n_splits - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  merge_split_partials<D, kWarps * 32, 4>(P.partials + pair * P.max_splits * pstride, n_splits, G,
                                      P.sinks ? P.sinks + kvh * G : nullptr, P.v_scale,
                                      P.out + ((int64_t)b * Hq + kvh * G) * D, P.tickets + pair,
                                      reinterpret_cast<float *>(smem), tid, CtaSync());
}

int max_keys_of(const Ctx &c, int layer, int max_seq_len) {
  const LayerInfo &L = c.layers[layer];
  int64_t mk = max_seq_len;
  if (L.kind == SWA_LAYER_SLIDING && L.window + 1 < mk) mk = L.window + 1;
  if (L.kind == SWA_LAYER_CHUNKED && L.window < mk) mk = L.window;
  return (int)(mk < 1 ? 1 : mk);
}

struct Layout {
  size_t part_off, total;
  int max_splits, split_keys;
};

Layout layout_of(const Ctx &c, int layer, int64_t nq, int max_seq_len) {
  Layout w;
  const LayerInfo &L = c.layers[layer];
  const int G = c.cfg.num_q_heads / L.hkv;
  const int mk = max_keys_of(c, layer, max_seq_len);
  w.split_keys = decode_split_keys(c.num_sms, nq, L.hkv, mk, c.cfg.page_size);
  w.max_splits = (mk + w.split_keys - 1) / w.split_keys;
  size_t part = (size_t)nq * L.hkv * w.max_splits * part_stride(G, c.cfg.head_dim) * sizeof(float);
  w.part_off = ws_partials_off(c, nq);
  w.total = w.part_off + (part + 255) / 256 * 256;
  return w;
}

template <int D, bool FP8, bool KM, int NW = 4>
cudaError_t launch_t(dim3 grid, const MmaParams &P, cudaStream_t s) {
  // Main tiles (or merge scratch), then the split's page-row table.
  const int smem = Smem<D, FP8, KM, NW>::kTotal + (P.split_keys / P.ps + 2) * (int)sizeof(int64_t);
  cudaError_t e = cudaFuncSetAttribute(k_decode_mma<D, FP8, KM, NW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: this grid may be scheduled while the
  // previous kernel on the stream finishes; the kernel waits for it before
  // its first global access, so stream order is kept.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_decode_mma<D, FP8, KM, NW>, P);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool mma_decode_supported(const Ctx &c, int layer) {
  if (c.cfg.kv_dtype != SWA_DTYPE_BF16 && c.cfg.kv_dtype != SWA_DTYPE_E4M3) return false;
  if (c.cfg.head_dim != 64 && c.cfg.head_dim != 128) return false;
  const int G = c.cfg.num_q_heads / c.layers[layer].hkv;
  return G >= 1 && G <= 16;
}

size_t mma_decode_ws_bytes(const Ctx &c, int layer, int64_t nq, int max_seq_len) {
  return layout_of(c, layer, nq, max_seq_len).total;
}

cudaError_t launch_attn_decode_mma(Ctx &c, const AttnArgs &a, cudaStream_t s) {
  if (a.nq == 0) return cudaSuccess;
  const LayerInfo &L = c.layers[a.layer];
  Layout w = layout_of(c, a.layer, a.nq, a.max_seq_len);
  MmaParams P;
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
  P.seq = a.seq;
  P.plan = a.plan;
  P.q = static_cast<const __nv_bfloat16 *>(a.q);
  P.sinks = a.sinks;
  const bool fp8 = c.cfg.kv_dtype == SWA_DTYPE_E4M3;
  P.qk_scale_log2 = a.scale * 1.4426950408889634f * (fp8 ? a.k_scale : 1.f);
  P.v_scale = fp8 ? a.v_scale : 1.f;
  P.out = static_cast<__nv_bfloat16 *>(a.out);
  P.partials = reinterpret_cast<float *>(static_cast<char *>(a.ws) + w.part_off);
  P.tickets = reinterpret_cast<int32_t *>(static_cast<char *>(a.ws) + 256);
  P.max_splits = w.max_splits;
  P.split_keys = w.split_keys;
  P.err = c.err_word;
  P.k_new = static_cast<const char *>(a.k_new);
  P.v_new = static_cast<const char *>(a.v_new);
  P.full_loc = a.full_loc;
  P.swa_loc = a.swa_loc;
  P.mapping = c.mapping;
  P.map_len = c.mapping_len;
  P.in_full = L.in_full ? 1 : 0;
  P.st_k_scale = a.k_scale;
  P.st_v_scale = a.v_scale;
  if (w.max_splits > 65535) return cudaErrorInvalidConfiguration;   // grid z limit
  dim3 grid(L.hkv, a.nq, w.max_splits);
  const int D = c.cfg.head_dim;
  if (P.G <= 8 && max_keys_of(c, a.layer, a.max_seq_len) <= 512) {
    // Short streams (sliding windows): two warps on 32-key stages, so that
    // more CTAs fit per SM and a whole layer runs in about one wave.
    if (D == 128) return fp8 ? launch_t<128, true, true, 2>(grid, P, s) : launch_t<128, false, true, 2>(grid, P, s);
    return fp8 ? launch_t<64, true, true, 2>(grid, P, s) : launch_t<64, false, true, 2>(grid, P, s);
  }
  if (P.G <= 8) {   // keys as rows
    if (D == 128) return fp8 ? launch_t<128, true, true>(grid, P, s) : launch_t<128, false, true>(grid, P, s);
    return fp8 ? launch_t<64, true, true>(grid, P, s) : launch_t<64, false, true>(grid, P, s);
  }
  if (D == 128) return fp8 ? launch_t<128, true, false>(grid, P, s) : launch_t<128, false, false>(grid, P, s);
  return fp8 ? launch_t<64, true, false>(grid, P, s) : launch_t<64, false, false>(grid, P, s);
}

}  // namespace swa
