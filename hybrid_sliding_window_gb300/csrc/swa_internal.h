// Internal declarations shared by the libswa translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "swa.h"

namespace swa {

constexpr int kMaxHeadDim = 256;

// One NVTX range per C-ABI call, named after the entry point, so a profiler
// timeline groups each call's launches (a no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};
#define SWA_NVTX(name) ::swa::NvtxRange swa_nvtx_range_(name)

// One free-page ledger on the device: a ring of page ids (front at head),
// a staging list (need_sort) and three counters in the state blob.
struct PoolDev {
  int64_t *ring;
  int64_t *staged;
  int64_t *head;
  int64_t *count;
  int64_t *nstaged;
  int64_t cap;        // number of pages of the pool (pages 1..cap)
  // SWA pool in per-request ring mode: slots of one ring (0: paged pool) and
  // the number of request slots; the ring of slot r starts at ps + r * ring_cost.
  int64_t ring_cost = 0;
  int64_t ring_slots = 0;
};

// Where the rows of one layer live.  Row of slot t:
//   per-layer: t;  envelope: (t / ps) * (ps * blocks) + t % ps.
struct KvAddr {
  char *k;            // per-layer: K array; envelope: raw + (2l) * ps * row_bytes
  char *v;            // per-layer: V array; envelope: raw + (2l+1) * ps * row_bytes
  int64_t row_bytes;  // Hkv * D * element size
  int32_t ps;
  int32_t blocks;     // envelope: 2 * layers of the pool; per-layer: 0
};

__host__ __device__ inline int64_t kv_row(const KvAddr &a, int64_t t) {
  if (a.blocks == 0) return t;
  return (t / a.ps) * ((int64_t)a.ps * a.blocks) + t % a.ps;
}

struct LayerInfo {
  int kind;
  int window;
  int hkv;
  int pool_layer;
  bool in_full;
  KvAddr addr;
  bool tma = false;       // TMA tensor maps below are valid
  CUtensorMap tmk, tmv;   // per-layer K / V as [rows][Hkv][D], box {64, 1, ps}
};

// Batch scratch in the state blob used by the eviction pass.
struct EvictScratch {
  int64_t *old_pos;
  int64_t *new_pos;
  int64_t *npages;   // pages of the range [old, new)
  int64_t *nlive;    // of those, pages that still hold a live SWA page
};

// Plan workspace layout: header int32 [bs][4] = {lo, hi, first_page, n_pages},
// then page ids int32 [bs][max_pages].
struct PlanView {
  const int32_t *hdr;
  const int32_t *pages;
  int32_t max_pages;
};

struct Ctx {
  swa_config cfg{};
  std::vector<swa_layer> layer_copy;
  std::vector<LayerInfo> layers;
  int L_full = 0, L_swa = 0;
  int lookback = 0;          // largest lookback of SWA-pool layers
  int64_t ring_cost = 0;     // per-request SWA ring slots (0: paged SWA pool)
  int32_t ring_slots = 0;
  int esize = 2;             // bytes per stored element
  int64_t np_full = 0, np_swa = 0;
  int64_t mapping_len = 0;
  // device state
  int64_t *mapping = nullptr;
  int64_t *counters = nullptr;
  PoolDev full{}, swa{};
  EvictScratch ev{};
  int32_t *err_word = nullptr;  // aliases counters[SWA_CTR_ERROR]
  // host mirrors, in pages
  int64_t h_count_full = 0, h_staged_full = 0, h_count_swa = 0, h_staged_swa = 0;
  std::string err;
  int last_path = -1;
  int num_sms = 0;
  int device = 0;
};

// ---- split workspace of the attention kernels -----------------------------
// [256 B reserved: work counters][tickets][partials].  The ticket block has
// one size for every layer and every decode batch of a context (max(nq,
// max_batch) x the largest KV-head count, int32), so decode calls of any
// layers can share one workspace: the partials of one layer never cover the
// tickets of another, which are zero between launches.
inline size_t ws_tickets_bytes(const Ctx &c, int64_t nq) {
  int hmax = 1;
  for (const LayerInfo &L : c.layers) hmax = L.hkv > hmax ? L.hkv : hmax;
  const int64_t n = nq > c.cfg.max_batch ? nq : c.cfg.max_batch;
  return ((size_t)n * hmax * sizeof(int32_t) + 255) / 256 * 256;
}
inline size_t ws_partials_off(const Ctx &c, int64_t nq) { return 256 + ws_tickets_bytes(c, nq); }
// Leading bytes of a decode workspace that must be zero before a launch (the
// counters and tickets; the kernels write every partial before reading it).
size_t decode_ws_zero_bytes(const swa_ctx *ctx, int64_t bs);

// ---- launchers (alloc.cu) -------------------------------------------------
cudaError_t launch_init_state(Ctx &c, const int64_t *init_full,
                              const int64_t *init_swa, cudaStream_t s);
cudaError_t launch_alloc_extend(Ctx &c, int bs, const int64_t *pre,
                                const int64_t *seq, const int64_t *last_loc,
                                int64_t *out_full, int64_t *out_swa,
                                int32_t *rt, int64_t rt_stride,
                                const int64_t *req_idx, int max_new,
                                cudaStream_t s);
cudaError_t launch_alloc_pages(Ctx &c, int64_t need, int64_t *out_full,
                               int64_t *out_swa, cudaStream_t s);
cudaError_t launch_merge_sorted(Ctx &c, bool full_pool, cudaStream_t s);
cudaError_t launch_release(Ctx &c, const int64_t *idx, int64_t n, bool do_full,
                           int64_t expect_full, int64_t expect_swa,
                           cudaStream_t s);
cudaError_t launch_evict(Ctx &c, int bs, const int32_t *rt, int64_t rt_stride,
                         const int64_t *req_idx, const int64_t *pre,
                         int64_t *evicted, const int64_t *prot, int interval,
                         int radix, cudaStream_t s);
cudaError_t launch_translate(Ctx &c, const int64_t *full_loc, int64_t n,
                             int64_t *swa_loc, cudaStream_t s);
cudaError_t launch_translate_for_kernel(const int64_t *v2p, int64_t n_pages,
                                       const int64_t *virt, int64_t n, int64_t ps,
                                       int64_t multiplier, int64_t *out, int32_t *err,
                                       int sms, cudaStream_t s);

// ---- store.cu ---------------------------------------------------------------
cudaError_t launch_store(Ctx &c, int layer, const void *k, const void *v,
                         int64_t n, const int64_t *full_loc,
                         const int64_t *swa_loc, float ks, float vs,
                         cudaStream_t s);

// ---- plan.cu ----------------------------------------------------------------
int plan_max_pages(const Ctx &c, int max_new);
cudaError_t launch_plan(Ctx &c, int bs, const int32_t *rt, int64_t rt_stride,
                        const int64_t *req_idx, const int64_t *pre,
                        const int64_t *seq, int max_new, void *plan,
                        cudaStream_t s);

// ---- attention ----------------------------------------------------------------
// Query description shared by decode and extend.
struct AttnArgs {
  int layer;
  int nq;                     // number of queries (decode: bs)
  int bs;
  const int32_t *rt;
  int64_t rt_stride;
  const int64_t *req_idx;
  const int64_t *pre;         // extend only
  const int64_t *seq;
  const int64_t *qo_indptr;   // extend only (NULL = decode)
  int max_seq_len;
  int max_new;
  PlanView plan;
  const void *q;
  const float *sinks;
  float scale;
  float k_scale, v_scale;
  void *out;
  void *ws;
  size_t ws_bytes;
  // Decode only, optional: the batch's new K/V rows ([bs][Hkv][D] bf16),
  // stored at their slots by the attention launch itself before it reads them.
  const void *k_new, *v_new;
  const int64_t *full_loc, *swa_loc;
};

size_t simt_ws_bytes(const Ctx &c, int layer, int64_t nq, int max_seq_len);
cudaError_t launch_attn_simt(Ctx &c, const AttnArgs &a, cudaStream_t s);

bool mma_decode_supported(const Ctx &c, int layer);
size_t mma_decode_ws_bytes(const Ctx &c, int layer, int64_t nq, int max_seq_len);
cudaError_t launch_attn_decode_mma(Ctx &c, const AttnArgs &a, cudaStream_t s);

bool tc_extend_supported(const Ctx &c, int layer);
// Builds the TMA tensor maps of one layer's K and V rows (bf16 or 8-bit,
// 128- or 256-byte head rows, page size 16..128); leaves tma = false when the
// layer does not qualify or encoding fails.
void make_kv_tensor_maps(Ctx &c, int layer);
// TMA tensor map over an extend call's queries or outputs, x [nq][hq][d]
// (bf16), whose box is one tile of up to 128 rows: {64 dims, g heads,
// 128 / g tokens}, 128-byte swizzle.  False if x is not 16-byte aligned, g is
// outside 1..128 or encoding fails.
bool make_qo_tensor_map(CUtensorMap *m, const void *x, int64_t nq, int hq, int d, int g);
size_t tc_extend_ws_bytes(const Ctx &c, int layer, int64_t n_tokens, int max_seq_len);
cudaError_t launch_attn_extend_tc(Ctx &c, const AttnArgs &a, cudaStream_t s);

// Records a message for swa_last_error(ctx) (defined in ctx.cu).
void set_ctx_error(swa_ctx *ctx, const char *msg);

// Device-side error helper.
__device__ inline void set_error(int32_t *word, int bits) {
  if (word) atomicOr(word, bits);
}

}  // namespace swa
