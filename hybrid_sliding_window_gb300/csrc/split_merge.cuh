// Split-KV bookkeeping shared by the tensor-core decode kernels: the partial
// layout in the workspace, the split size, and the merge that the last split
// of a (request, KV head) runs.
//
// Method: "SWA in SGLang" design note - a per-head sink logit joins the
// softmax denominator; splitting the keys of one query row and merging the
// per-split (max, sum, unnormalised output) is exact up to rounding, the
// usual log-sum-exp rescaling.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace swa {

// Partials of one split: the G x D unnormalised output rows, then (max, sum)
// per row; the stride is padded to whole float4s so the merge reads 16 bytes
// at a time.
__host__ __device__ inline int part_stride(int G, int D) { return (G * D + 2 * G + 3) & ~3; }

// Keys per split.  A split is one CTA's (or one persistent work item's) run
// of the key stream; each costs a fixed prologue (page rows, first tiles in
// flight) and epilogue (warp merge, partial write, ticket) of several
// microseconds, so long splits pay less; but the last splits to start set the
// tail, so they must stay short against the per-SM share of the work.  Only
// the batch and the longest request are known on the host: the longest
// request gets about eight splits (a power of two from 1024 to 4096 keys),
// halved while there are fewer than two splits per SM slot (2 CTAs per SM,
// counted for a mean of half the longest request), down to 1024; at most 512
// pages per split (the page-row table lives in shared memory).
inline int decode_split_keys(int num_sms, int64_t nq, int hkv, int64_t max_keys, int ps) {
  const int64_t slots = 2LL * (num_sms > 0 ? num_sms : 148);
  int split = 1024;
  while (split < 4096 && split * 8LL < max_keys) split *= 2;
  while (split > 1024 && nq * hkv * ((max_keys / 2 + split - 1) / split) < 2 * slots) split /= 2;
  return split < 512 * ps ? split : 512 * ps;
}

constexpr int kMergeChunk = 256;   // split weights staged per pass
// Shared-memory bytes the merge needs (weights of 16 rows, row maxima, scales).
constexpr int kMergeScratchBytes = (16 * kMergeChunk + 32) * 4;

// Merge of the n_splits partials of one (request, KV head), run by the
// kThreads threads (tid 0..kThreads-1) of the split that finished last.
// Row statistics first (one warp per query row; the sink joins the
// denominator), then the weighted sum of the output blocks: each thread owns
// up to four float4 columns and keeps the loads of several splits in
// flight.  `sync` is the barrier over those threads; `out` points at the G
// output rows of this (request, KV head); `sinks` at its G sink logits or
// null.  kUnroll splits are read per step of the sum (their loads in flight
// together).  The ticket is reset for the next launch.
template <int D, int kThreads, int kUnroll, class Sync>
__device__ __forceinline__ void merge_split_partials(const float *base, int n_splits, int G,
                                                     const float *sinks, float v_scale,
                                                     __nv_bfloat16 *out, int32_t *ticket,
                                                     float *scratch, int tid, Sync sync) {
  constexpr int kWarpsM = kThreads / 32;
  const int warp = tid >> 5, lane = tid & 31;
  const int pstride = part_stride(G, D);
  float *s_w = scratch;                 // [16][kMergeChunk]
  float *s_mf = s_w + 16 * kMergeChunk; // [16] merged row maxima (log2 domain)
  float *s_il = s_mf + 16;              // [16] v_scale / denominator
  for (int gg = warp; gg < G; gg += kWarpsM) {
    const float *ml = base + G * D + 2 * gg;
    float mx = -INFINITY;
    for (int s = lane; s < n_splits; s += 32) mx = fmaxf(mx, __ldcg(ml + (int64_t)s * pstride));
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float Mf = mx, extra = 0.f;
    if (sinks) {
      const float sg = sinks[gg] * 1.4426950408889634f;
      Mf = fmaxf(mx, sg);
      extra = exp2f(sg - Mf);
    }
    float L = 0.f;
    for (int s = lane; s < n_splits; s += 32) {
      const float *q = ml + (int64_t)s * pstride;
      L += exp2f(__ldcg(q) - Mf) * __ldcg(q + 1);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      s_mf[gg] = Mf;
      s_il[gg] = v_scale / (L + extra);
    }
  }
  sync();
  constexpr int kQuads = D / 4;
  constexpr int kPer = (16 * kQuads + kThreads - 1) / kThreads;
  float4 acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < n_splits; c0 += kMergeChunk) {
    const int cn = min(kMergeChunk, n_splits - c0);
    for (int i = tid; i < G * cn; i += kThreads) {
      const int gg = i / cn, s = i - gg * cn;
      s_w[gg * kMergeChunk + s] =
          exp2f(__ldcg(base + (int64_t)(c0 + s) * pstride + G * D + 2 * gg) - s_mf[gg]);
    }
    sync();
    const float4 *blk = reinterpret_cast<const float4 *>(base + (int64_t)c0 * pstride);
#pragma unroll kUnroll
    for (int s = 0; s < cn; ++s) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int f = tid + i * kThreads;
        if (f < G * kQuads) {
          const float4 v = __ldcg(blk + (int64_t)s * (pstride / 4) + f);
          const float w = s_w[(f / kQuads) * kMergeChunk + s];
          acc[i].x += w * v.x;
          acc[i].y += w * v.y;
          acc[i].z += w * v.z;
          acc[i].w += w * v.w;
        }
      }
    }
    sync();
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int f = tid + i * kThreads;
    if (f < G * kQuads) {
      const int gg = f / kQuads, d = (f % kQuads) * 4;
      const float il = s_il[gg];
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * il, acc[i].y * il);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * il, acc[i].w * il);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t *>(&lo);
      w.y = *reinterpret_cast<uint32_t *>(&hi);
      *reinterpret_cast<uint2 *>(out + (int64_t)gg * D + d) = w;
    }
  }
  if (tid == 0) *ticket = 0;
}

}  // namespace swa
