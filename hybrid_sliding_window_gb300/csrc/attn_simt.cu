// Generic paged attention on CUDA cores: any stored dtype (f32 / bf16 / e4m3),
// any page size, both KV layouts, decode and extend.  It is the reference
// GPU path every configuration can take; tensor-core kernels cover the hot
// configurations.
//
// Method ("SWA in SGLang" design note, "problem", "design" and "which
// models, which layers"): query at position p, query head h reads KV head
// h / G; keys J = 0..p (full), max(0, p - Wx)..p (sliding, Wx excludes the
// current token) or floor(p / C) * C..p (chunked local); a per-head sink
// logit joins the softmax denominator only.
//
// Work item = (query, KV head, split of SPLIT keys).  A CTA first looks up
// the KV rows of all keys of its split (one independent load per key, all
// threads), then 4 warps each walk every 4th key keeping one online-softmax
// state for the G query heads of its KV head (scores in log2 units), with the
// K/V rows of their next 4 keys loaded before any is used; it merges the
// warps in shared memory, and either
// writes the output (one split) or a partial (m, l, acc); the last CTA of a
// (query, KV head) to finish - found with an atomic ticket - merges the
// partials, folds in the sink and resets the ticket, so one launch does both.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include "swa_internal.h"

namespace swa {
namespace {

constexpr int kWarps = 4;
constexpr int kSplit = 512;      // longest split (the row table in shared memory)
constexpr int kMinSplit = 32;
constexpr int kGMax = 16;
constexpr float kNegBig = -1e30f;

struct SimtParams {
  int kind, window, hkv, G, D, ps;
  KvAddr addr;
  int64_t pool_rows;
  const int32_t *rt;
  int64_t rt_stride;
  const int64_t *req_idx;
  const int64_t *pre;
  const int64_t *seq;
  const int64_t *qo_indptr;
  int bs;
  PlanView plan;
  const void *q;
  const float *sinks;
  float scale_log2;
  float k_scale, v_scale;
  void *out;
  float *partials;
  int32_t *tickets;
  int max_splits;
  int split_keys;             // keys per split, a power of two in [kMinSplit, kSplit]
  int32_t *err;
};

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ inline float get(const float *p, int i) { return p[i]; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ inline float get(const __nv_bfloat16 *p, int i) { return __bfloat162float(p[i]); }
};
template <> struct Elem<__nv_fp8_e4m3> {
  static __device__ inline float get(const __nv_fp8_e4m3 *p, int i) { return float(p[i]); }
};

template <typename QT> __device__ inline float qload(const QT *p, int64_t i);
template <> __device__ inline float qload<float>(const float *p, int64_t i) { return p[i]; }
template <> __device__ inline float qload<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
  return __bfloat162float(p[i]);
}
template <typename QT> __device__ inline void ostore(QT *p, int64_t i, float v);
template <> __device__ inline void ostore<float>(float *p, int64_t i, float v) { p[i] = v; }
template <> __device__ inline void ostore<__nv_bfloat16>(__nv_bfloat16 *p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// Locate query i: its batch entry b and position p.
__device__ inline void locate_query(const SimtParams &P, int i, int &b, int64_t &p) {
  if (!P.qo_indptr) {
    b = i;
    p = P.seq[i] - 1;
    return;
  }
  int lo = 0, hi = P.bs;  // find b with indptr[b] <= i < indptr[b+1]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (P.qo_indptr[mid] <= i) lo = mid; else hi = mid;
  }
  b = lo;
  p = P.pre[b] + (i - P.qo_indptr[b]);
}

__device__ inline int64_t key_lo(int kind, int window, int64_t p) {
  if (kind == SWA_LAYER_FULL) return 0;
  if (kind == SWA_LAYER_SLIDING) return p - window > 0 ? p - window : 0;
  return (p / window) * window;
}

// Slot of position j of batch entry b on this layer.
__device__ inline int64_t slot_of(const SimtParams &P, int b, int64_t j) {
  if (P.kind == SWA_LAYER_FULL) {
    return P.rt[P.req_idx[b] * P.rt_stride + j];
  }
  const int32_t *h = P.plan.hdr + b * 4;
  int64_t k = j / P.ps - h[2];
  if (j < h[0] || k < 0 || k >= h[3]) {
    set_error(P.err, SWA_DEVERR_RANGE);
    return 0;
  }
  int64_t page = P.plan.pages[(int64_t)b * P.plan.max_pages + k];
  if (page <= 0) set_error(P.err, SWA_DEVERR_WINDOW_EVICTED);
  return page * P.ps + j % P.ps;
}

template <typename KT, typename QT, int DL>
__global__ void __launch_bounds__(kWarps * 32) k_attn_simt(SimtParams P) {
  constexpr int D = DL * 32;
  const int split = blockIdx.x, kvh = blockIdx.y, qi = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = P.G;
  int b;
  int64_t p;
  locate_query(P, qi, b, p);
  const int64_t lo = key_lo(P.kind, P.window, p);
  const int64_t n_keys = p - lo + 1;
  const int n_splits = (int)((n_keys + P.split_keys - 1) / P.split_keys);
  if (split >= n_splits) return;
  const int64_t k0 = lo + (int64_t)split * P.split_keys;
  const int64_t k1 = min(p + 1, k0 + P.split_keys);

  __shared__ float qs[kGMax][D];
  __shared__ float sm_m[kWarps][kGMax], sm_l[kWarps][kGMax];
  __shared__ float sm_acc[kWarps][kGMax][D];
  __shared__ int64_t s_row[kSplit];
  __shared__ int s_last;

  const QT *qp = static_cast<const QT *>(P.q);
  const int Hq = P.hkv * G;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    int g = e / D, d = e % D;
    qs[g][d] = qload<QT>(qp, ((int64_t)qi * Hq + kvh * G + g) * D + d) * P.scale_log2;
  }
  // KV rows of the split's keys, looked up once (independent loads).
  const int nk = (int)(k1 - k0);
  for (int i = threadIdx.x; i < nk; i += blockDim.x) {
    int64_t slot = slot_of(P, b, k0 + i);
    if (slot < 0 || slot >= P.pool_rows) {
      set_error(P.err, SWA_DEVERR_RANGE);
      slot = 0;
    }
    s_row[i] = kv_row(P.addr, slot);
  }
  __syncthreads();

  float m[kGMax], l[kGMax], acc[kGMax][DL];
#pragma unroll
  for (int g = 0; g < kGMax; ++g) {
    m[g] = kNegBig;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[g][e] = 0.f;
  }
  const float ksc = P.k_scale, vsc = P.v_scale;
  constexpr int kAhead = 4;   // keys of one warp whose K/V rows are in flight together
  for (int i0 = warp; i0 < nk; i0 += kWarps * kAhead) {
    float kf[kAhead][DL], vf[kAhead][DL];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int i = i0 + u * kWarps;
      if (i < nk) {
        const int64_t row = s_row[i];
        const KT *kr = reinterpret_cast<const KT *>(P.addr.k + row * P.addr.row_bytes) + kvh * D + lane * DL;
        const KT *vr = reinterpret_cast<const KT *>(P.addr.v + row * P.addr.row_bytes) + kvh * D + lane * DL;
#pragma unroll
        for (int e = 0; e < DL; ++e) {
          kf[u][e] = Elem<KT>::get(kr, e) * ksc;
          vf[u][e] = Elem<KT>::get(vr, e) * vsc;
        }
      } else {
#pragma unroll
        for (int e = 0; e < DL; ++e) kf[u][e] = vf[u][e] = 0.f;
      }
    }
    // Scores of the keys first (independent reductions, in flight
    // together), then the online-softmax updates in key order.
    float sc[kAhead][kGMax];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
#pragma unroll
      for (int g = 0; g < kGMax; ++g) {
        if (g < G) {
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < DL; ++e) s += qs[g][lane * DL + e] * kf[u][e];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          sc[u][g] = s;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      if (i0 + u * kWarps >= nk) break;
#pragma unroll
      for (int g = 0; g < kGMax; ++g) {
        if (g < G) {
          const float s = sc[u][g];
          float mn = fmaxf(m[g], s);
          float corr = exp2f(m[g] - mn);
          float pe = exp2f(s - mn);
          l[g] = l[g] * corr + pe;
#pragma unroll
          for (int e = 0; e < DL; ++e) acc[g][e] = acc[g][e] * corr + pe * vf[u][e];
          m[g] = mn;
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < kGMax; ++g) {
    if (g < G) {
      if (lane == 0) { sm_m[warp][g] = m[g]; sm_l[warp][g] = l[g]; }
#pragma unroll
      for (int e = 0; e < DL; ++e) sm_acc[warp][g][lane * DL + e] = acc[g][e];
    }
  }
  __syncthreads();

  // Merge the warps: state of this split per (g, d).
  QT *op = static_cast<QT *>(P.out);
  const bool single = n_splits == 1;
  const int64_t item = ((int64_t)qi * P.hkv + kvh) * P.max_splits + split;
  const int stride = G * (D + 2);
  float *part = P.partials + item * stride;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    int g = e / D, d = e % D;
    float M = kNegBig;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][g]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      float f = exp2f(sm_m[w][g] - M);
      L += sm_l[w][g] * f;
      A += sm_acc[w][g][d] * f;
    }
    if (single) {
      float Mf = M, extra = 0.f;
      if (P.sinks) {
        float sg = P.sinks[kvh * G + g] * 1.4426950408889634f;
        Mf = fmaxf(M, sg);
        extra = exp2f(sg - Mf);
      }
      float r = exp2f(M - Mf);
      ostore<QT>(op, ((int64_t)qi * Hq + kvh * G + g) * D + d, A * r / (L * r + extra));
    } else {
      part[g * (D + 2) + 2 + d] = A;
      if (d == 0) { part[g * (D + 2)] = M; part[g * (D + 2) + 1] = L; }
    }
  }
  if (single) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int prev = atomicAdd(&P.tickets[(int64_t)qi * P.hkv + kvh], 1);
    s_last = (prev == n_splits - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float *base = P.partials + ((int64_t)qi * P.hkv + kvh) * P.max_splits * stride;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    int g = e / D, d = e % D;
    float M = kNegBig;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, __ldcg(base + s * stride + g * (D + 2)));
    float Mf = M, extra = 0.f;
    if (P.sinks) {
      float sg = P.sinks[kvh * G + g] * 1.4426950408889634f;
      Mf = fmaxf(M, sg);
      extra = exp2f(sg - Mf);
    }
    float L = extra, A = 0.f;
    for (int s = 0; s < n_splits; ++s) {
      const float *ps_ = base + s * stride + g * (D + 2);
      float f = exp2f(__ldcg(ps_) - Mf);
      L += __ldcg(ps_ + 1) * f;
      A += __ldcg(ps_ + 2 + d) * f;
    }
    ostore<QT>(op, ((int64_t)qi * Hq + kvh * G + g) * D + d, A / L);
  }
  if (threadIdx.x == 0) P.tickets[(int64_t)qi * P.hkv + kvh] = 0;
}

int max_keys(const Ctx &c, int layer, int max_seq_len) {
  const LayerInfo &L = c.layers[layer];
  int64_t mk = max_seq_len;
  if (L.kind == SWA_LAYER_SLIDING && L.window + 1 < mk) mk = L.window + 1;
  if (L.kind == SWA_LAYER_CHUNKED && L.window < mk) mk = L.window;
  return (int)(mk < 1 ? 1 : mk);
}

struct WsLayout {
  size_t partial_bytes;
  size_t part_off;
  size_t total;
  int max_splits;
  int split_keys;
};

WsLayout ws_layout(const Ctx &c, int layer, int64_t nq, int max_seq_len) {
  WsLayout w;
  const LayerInfo &L = c.layers[layer];
  const int G = c.cfg.num_q_heads / L.hkv;
  // Split size: the longest (kSplit) unless the launch would then fill less
  // than one wave of 2 CTAs per SM; small batches cut their keys finer so
  // more CTAs walk them in parallel (partials merged in the same launch).
  const int mk = max_keys(c, layer, max_seq_len);
  const int64_t slots = 2LL * (c.num_sms > 0 ? c.num_sms : 148);
  w.split_keys = kSplit;
  while (w.split_keys > kMinSplit &&
         nq * L.hkv * ((mk + w.split_keys - 1) / w.split_keys) < slots)
    w.split_keys /= 2;
  w.max_splits = (mk + w.split_keys - 1) / w.split_keys;
  w.partial_bytes = (size_t)nq * L.hkv * w.max_splits * G * (c.cfg.head_dim + 2) * sizeof(float);
  w.part_off = ws_partials_off(c, nq);   // [reserved][tickets][partials]
  w.total = w.part_off + (w.partial_bytes + 255) / 256 * 256;
  return w;
}

template <typename KT, typename QT>
cudaError_t dispatch_dl(int D, dim3 grid, const SimtParams &P, cudaStream_t s) {
  switch (D) {
    case 32: k_attn_simt<KT, QT, 1><<<grid, kWarps * 32, 0, s>>>(P); break;
    case 64: k_attn_simt<KT, QT, 2><<<grid, kWarps * 32, 0, s>>>(P); break;
    case 128: k_attn_simt<KT, QT, 4><<<grid, kWarps * 32, 0, s>>>(P); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

size_t simt_ws_bytes(const Ctx &c, int layer, int64_t nq, int max_seq_len) {
  return ws_layout(c, layer, nq, max_seq_len).total;
}

cudaError_t launch_attn_simt(Ctx &c, const AttnArgs &a, cudaStream_t s) {
  if (a.nq == 0) return cudaSuccess;
  const LayerInfo &L = c.layers[a.layer];
  WsLayout w = ws_layout(c, a.layer, a.nq, a.max_seq_len);
  SimtParams P;
  P.kind = L.kind;
  P.window = L.window;
  P.hkv = L.hkv;
  P.G = c.cfg.num_q_heads / L.hkv;
  P.D = c.cfg.head_dim;
  P.ps = c.cfg.page_size;
  P.addr = L.addr;
  P.pool_rows = (L.in_full ? c.cfg.size_full : c.cfg.size_swa) + c.cfg.page_size;
  P.rt = a.rt;
  P.rt_stride = a.rt_stride;
  P.req_idx = a.req_idx;
  P.pre = a.pre;
  P.seq = a.seq;
  P.qo_indptr = a.qo_indptr;
  P.bs = a.bs;
  P.plan = a.plan;
  P.q = a.q;
  P.sinks = a.sinks;
  P.scale_log2 = a.scale * 1.4426950408889634f;
  // Scales apply to decoded E4M3 values only.
  P.k_scale = c.cfg.kv_dtype == SWA_DTYPE_E4M3 ? a.k_scale : 1.f;
  P.v_scale = c.cfg.kv_dtype == SWA_DTYPE_E4M3 ? a.v_scale : 1.f;
  P.out = a.out;
  P.partials = reinterpret_cast<float *>(static_cast<char *>(a.ws) + w.part_off);
  P.tickets = reinterpret_cast<int32_t *>(static_cast<char *>(a.ws) + 256);
  P.max_splits = w.max_splits;
  P.split_keys = w.split_keys;
  P.err = c.err_word;
  dim3 grid(w.max_splits, L.hkv, a.nq);
  if (c.cfg.kv_dtype == SWA_DTYPE_F32) return dispatch_dl<float, float>(P.D, grid, P, s);
  if (c.cfg.kv_dtype == SWA_DTYPE_BF16)
    return dispatch_dl<__nv_bfloat16, __nv_bfloat16>(P.D, grid, P, s);
  return dispatch_dl<__nv_fp8_e4m3, __nv_bfloat16>(P.D, grid, P, s);
}

}  // namespace swa
