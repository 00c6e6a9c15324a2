// libswa C-ABI: configuration checks, the device state blob, host mirrors of
// the free counts, and dispatch to the kernels.  See include/swa.h for the
// contract of every entry point.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <string>

#include "swa_internal.h"

struct swa_ctx : public swa::Ctx {
  bool mirror_stale = false;
  int forced_path = -1;
};

namespace {

using swa::Ctx;

thread_local std::string g_create_err;
constexpr int64_t kMaxBitmapPages = 1700000;  // bitmap of a pool fits in shared memory

swa_status fail(swa_ctx *c, swa_status st, const std::string &msg) {
  if (c) c->err = msg;
  else g_create_err = msg;
  return st;
}

#define CUDA_TRY(c, expr)                                                        \
  do {                                                                           \
    cudaError_t e_ = (expr);                                                     \
    if (e_ != cudaSuccess)                                                       \
      return fail(c, SWA_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(e_)); \
  } while (0)

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t al256(size_t x) { return (x + 255) / 256 * 256; }

struct StateLayout {
  size_t counters, ev, mapping, ring_full, staged_full, ring_swa, staged_swa, total;
};

StateLayout state_layout(const swa_config *cfg) {
  StateLayout L;
  const int64_t ps = cfg->page_size;
  const int64_t npf = cfg->size_full / ps, nps = cfg->size_swa / ps;
  const int64_t map_len = cfg->size_full + ps + 1;
  size_t off = 0;
  L.counters = off; off = al256(off + 64 * sizeof(int64_t));
  L.ev = off; off = al256(off + 4 * (size_t)cfg->max_batch * sizeof(int64_t));
  L.mapping = off; off = al256(off + (size_t)map_len * sizeof(int64_t));
  L.ring_full = off; off = al256(off + (size_t)npf * sizeof(int64_t));
  L.staged_full = off; off = al256(off + (size_t)npf * sizeof(int64_t));
  L.ring_swa = off; off = al256(off + (size_t)nps * sizeof(int64_t));
  L.staged_swa = off; off = al256(off + (size_t)nps * sizeof(int64_t));
  L.total = off;
  return L;
}

int esize_of(int dtype) { return dtype == SWA_DTYPE_F32 ? 4 : dtype == SWA_DTYPE_BF16 ? 2 : 1; }

// Checks that need no device; fills the layer table.
swa_status check_config(const swa_config *cfg, Ctx &c) {
  if (!cfg || !cfg->layers) return fail(nullptr, SWA_ERR_INVALID, "null config or layers");
  if (cfg->num_layers < 1 || cfg->page_size < 1 || cfg->max_batch < 1)
    return fail(nullptr, SWA_ERR_CONFIG, "num_layers, page_size and max_batch must be >= 1");
  const int64_t ps = cfg->page_size;
  if (cfg->size_full < ps || cfg->size_swa < ps || cfg->size_full % ps || cfg->size_swa % ps)
    return fail(nullptr, SWA_ERR_CONFIG, "pool sizes must be positive multiples of page_size");
  if (cfg->head_dim != 32 && cfg->head_dim != 64 && cfg->head_dim != 128)
    return fail(nullptr, SWA_ERR_CONFIG, "head_dim must be 32, 64 or 128");
  if (cfg->kv_dtype < SWA_DTYPE_F32 || cfg->kv_dtype > SWA_DTYPE_E4M3)
    return fail(nullptr, SWA_ERR_CONFIG, "unknown kv_dtype");
  if (cfg->layout != SWA_LAYOUT_PER_LAYER && cfg->layout != SWA_LAYOUT_ENVELOPE)
    return fail(nullptr, SWA_ERR_CONFIG, "unknown layout");
  if (cfg->num_q_heads < 1) return fail(nullptr, SWA_ERR_CONFIG, "num_q_heads < 1");
  if (cfg->size_full / ps > kMaxBitmapPages || cfg->size_swa / ps > kMaxBitmapPages)
    return fail(nullptr, SWA_ERR_CONFIG, "a pool has more pages than the release bitmap holds");
  c.esize = esize_of(cfg->kv_dtype);
  c.layers.clear();
  int hkv_pool[2] = {-1, -1};
  c.L_full = c.L_swa = 0;
  c.lookback = 0;
  for (int l = 0; l < cfg->num_layers; ++l) {
    const swa_layer &s = cfg->layers[l];
    swa::LayerInfo L{};
    L.kind = s.kind;
    L.window = s.window;
    L.hkv = s.num_kv_heads;
    if (s.kind < SWA_LAYER_FULL || s.kind > SWA_LAYER_CHUNKED)
      return fail(nullptr, SWA_ERR_CONFIG, "layer " + std::to_string(l) + ": unknown kind");
    if (s.num_kv_heads < 1 || cfg->num_q_heads % s.num_kv_heads)
      return fail(nullptr, SWA_ERR_CONFIG, "layer " + std::to_string(l) + ": Hq % Hkv != 0");
    if (cfg->num_q_heads / s.num_kv_heads > 16)
      return fail(nullptr, SWA_ERR_CONFIG, "layer " + std::to_string(l) + ": GQA group > 16");
    if ((s.kind == SWA_LAYER_SLIDING && s.window < 0) || (s.kind == SWA_LAYER_CHUNKED && s.window < 1))
      return fail(nullptr, SWA_ERR_CONFIG, "layer " + std::to_string(l) + ": bad window");
    if (((int64_t)s.num_kv_heads * cfg->head_dim * c.esize) % 16)
      return fail(nullptr, SWA_ERR_CONFIG, "row bytes must be a multiple of 16");
    L.in_full = s.kind == SWA_LAYER_FULL;
    L.pool_layer = L.in_full ? c.L_full++ : c.L_swa++;
    if (!L.in_full) {
      int lb = s.kind == SWA_LAYER_SLIDING ? s.window : s.window - 1;
      c.lookback = std::max(c.lookback, lb);
    }
    int &h = hkv_pool[L.in_full ? 0 : 1];
    if (cfg->layout == SWA_LAYOUT_ENVELOPE && h != -1 && h != s.num_kv_heads)
      return fail(nullptr, SWA_ERR_CONFIG, "envelope pool layers must share num_kv_heads");
    h = s.num_kv_heads;
    if (cfg->layout == SWA_LAYOUT_PER_LAYER && (!s.k || !s.v))
      return fail(nullptr, SWA_ERR_INVALID, "layer " + std::to_string(l) + ": null K/V");
    c.layers.push_back(L);
  }
  if (cfg->swa_ring_size < 0 || cfg->ring_slots < 0)
    return fail(nullptr, SWA_ERR_CONFIG, "negative swa_ring_size or ring_slots");
  c.ring_cost = 0;
  c.ring_slots = 0;
  if (cfg->swa_ring_size > 0) {
    // Per-request rings: one ring of ceil(ring / ps) * ps slots per request slot.
    const int64_t cost = cdiv(cfg->swa_ring_size, ps) * ps;
    if (cfg->ring_slots < 1) return fail(nullptr, SWA_ERR_CONFIG, "ring mode needs ring_slots >= 1");
    if (cfg->swa_ring_size < (int64_t)c.lookback + 1)
      return fail(nullptr, SWA_ERR_CONFIG, "swa_ring_size is smaller than the window");
    if (cfg->size_swa != (int64_t)cfg->ring_slots * cost)
      return fail(nullptr, SWA_ERR_CONFIG, "ring mode: size_swa must equal ring_slots * ring cost");
    c.ring_cost = cost;
    c.ring_slots = cfg->ring_slots;
  } else if (c.L_swa > 0 && cfg->size_swa <= (int64_t)c.lookback + ps) {
    return fail(nullptr, SWA_ERR_CONFIG, "SWA pool cannot hold one request (N_swa <= W + P)");
  }
  // Row addressing.
  for (int l = 0; l < cfg->num_layers; ++l) {
    swa::LayerInfo &L = c.layers[l];
    const int64_t row_bytes = (int64_t)L.hkv * cfg->head_dim * c.esize;
    L.addr.row_bytes = row_bytes;
    L.addr.ps = cfg->page_size;
    if (cfg->layout == SWA_LAYOUT_PER_LAYER) {
      L.addr.k = static_cast<char *>(cfg->layers[l].k);
      L.addr.v = static_cast<char *>(cfg->layers[l].v);
      L.addr.blocks = 0;
    } else {
      const int Lp = L.in_full ? c.L_full : c.L_swa;
      char *raw = static_cast<char *>(L.in_full ? cfg->full_envelope : cfg->swa_envelope);
      const int64_t bytes = L.in_full ? cfg->full_envelope_bytes : cfg->swa_envelope_bytes;
      if (!raw) return fail(nullptr, SWA_ERR_INVALID, "null envelope buffer");
      const int64_t pages = (L.in_full ? cfg->size_full : cfg->size_swa) / ps + 1;
      const int64_t n_rows = pages * 2 * Lp * ps;
      if (n_rows >= (int64_t(1) << 31))
        return fail(nullptr, SWA_ERR_CONFIG, "envelope row ids overflow int32 (n_rows >= 2^31)");
      const int64_t last_view_end = ((2 * (int64_t)Lp - 1) * ps + n_rows) * row_bytes;
      if (last_view_end > bytes)
        return fail(nullptr, SWA_ERR_CONFIG, "envelope buffer lacks the one-envelope tail pad");
      L.addr.k = raw + (int64_t)(2 * L.pool_layer) * ps * row_bytes;
      L.addr.v = raw + (int64_t)(2 * L.pool_layer + 1) * ps * row_bytes;
      L.addr.blocks = 2 * Lp;
    }
  }
  return SWA_OK;
}

bool ensure_pages(swa_ctx *c, bool full, int64_t n, cudaStream_t s) {
  int64_t &cnt = full ? c->h_count_full : c->h_count_swa;
  int64_t &st = full ? c->h_staged_full : c->h_staged_swa;
  if (c->cfg.need_sort && n > cnt && st > 0) {
    if (swa::launch_merge_sorted(*c, full, s) != cudaSuccess) return false;
    cnt += st;
    st = 0;
  }
  return n <= cnt;
}

void mirror_release(swa_ctx *c, bool full, int64_t pages) {
  if (pages < 0) {
    c->mirror_stale = true;
    return;
  }
  if (c->cfg.need_sort) (full ? c->h_staged_full : c->h_staged_swa) += pages;
  else (full ? c->h_count_full : c->h_count_swa) += pages;
}

swa::PlanView plan_view(const swa_ctx *c, const void *plan, int bs, int max_new) {
  swa::PlanView v;
  v.hdr = static_cast<const int32_t *>(plan);
  v.pages = v.hdr ? v.hdr + (((int64_t)bs * 4 + 63) / 64) * 64 : nullptr;
  v.max_pages = swa::plan_max_pages(*c, max_new);
  return v;
}

}  // namespace

void swa::set_ctx_error(swa_ctx *ctx, const char *msg) {
  if (ctx) ctx->err = msg;
}

size_t swa::decode_ws_zero_bytes(const swa_ctx *ctx, int64_t bs) {
  return ctx ? swa::ws_partials_off(*ctx, bs) : 0;
}

extern "C" {

swa_status swa_pool_sizes(int64_t mem_bytes, int64_t F, int64_t S, int32_t L_full,
                          int32_t L_swa, double r, int32_t page_size, int32_t window,
                          int64_t *n_full, int64_t *n_swa) {
  if (!n_full || !n_swa || page_size < 1 || F < 0 || S < 0 || r < 0)
    return fail(nullptr, SWA_ERR_INVALID, "bad sizing arguments");
  const double cell = (double)F * L_full + r * (double)S * L_swa;
  if (cell <= 0) return fail(nullptr, SWA_ERR_INVALID, "empty cell");
  int64_t nf = (int64_t)std::floor((double)mem_bytes / cell);
  int64_t ns = (int64_t)std::floor(r * (double)nf);
  nf = nf / page_size * page_size;
  ns = ns / page_size * page_size;
  *n_full = nf;
  *n_swa = ns;
  if (ns <= (int64_t)window + page_size)
    return fail(nullptr, SWA_ERR_CONFIG, "SWA pool cannot hold one request (N_swa <= W + P)");
  return SWA_OK;
}

swa_status swa_decode_alloc_sizes(int32_t algo, int32_t steps, int32_t topk,
                                  int32_t draft_tokens, int32_t has_draft_kv,
                                  int32_t page_size, int64_t *alloc_len, int64_t *reserve,
                                  int64_t *rt_extra) {
  if (!alloc_len || !reserve || !rt_extra || page_size < 1 || algo < SWA_SPEC_NONE ||
      algo > SWA_SPEC_UNO)
    return fail(nullptr, SWA_ERR_INVALID, "bad speculative sizing arguments");
  const int64_t ps = page_size;
  const int64_t d = draft_tokens > 0 ? draft_tokens : 0;
  int64_t len = 1;
  if (algo == SWA_SPEC_UNO) {
    if (draft_tokens < 0) return fail(nullptr, SWA_ERR_INVALID, "UNO needs draft_tokens");
    len = d + 1;
  } else if (algo == SWA_SPEC_DRAFT) {
    const int64_t s = steps > 1 ? steps : 1, k = topk > 1 ? topk : 1;
    if (ps == 1 || k == 1 || !has_draft_kv) {
      len = std::max(s * k, d);
    } else {
      const int64_t pages_per_branch = (ps - 1 + s + ps - 1) / ps;
      len = std::max(pages_per_branch * ps * k, d);
    }
  }
  *alloc_len = len;
  *reserve = 2 * len;
  int64_t extra = 4 + d;
  if (algo != SWA_SPEC_NONE && (ps > 1 || algo == SWA_SPEC_UNO))
    extra = std::max(extra, 2 * len + ps - 1);
  *rt_extra = extra;
  return SWA_OK;
}

size_t swa_state_bytes(const swa_config *cfg) {
  if (!cfg || cfg->page_size < 1 || cfg->max_batch < 1) return 0;
  return state_layout(cfg).total;
}

swa_status swa_ctx_create(const swa_config *cfg, void *state_dev, const int64_t *init_free_full,
                          const int64_t *init_free_swa, swa_stream_t stream, swa_ctx **out) {
  SWA_NVTX("swa_ctx_create");
  if (!out || !state_dev) return fail(nullptr, SWA_ERR_INVALID, "null state or output pointer");
  *out = nullptr;
  if (reinterpret_cast<uintptr_t>(state_dev) % 256)
    return fail(nullptr, SWA_ERR_INVALID, "state blob must be 256-byte aligned");
  swa_ctx *c = new (std::nothrow) swa_ctx();
  if (!c) return fail(nullptr, SWA_ERR_INVALID, "out of host memory");
  swa_status st = check_config(cfg, *c);
  if (st != SWA_OK) {
    delete c;
    return st;
  }
  c->cfg = *cfg;
  c->layer_copy.assign(cfg->layers, cfg->layers + cfg->num_layers);
  c->cfg.layers = c->layer_copy.data();
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e != cudaSuccess) {
    g_create_err = std::string("cuda device query: ") + cudaGetErrorString(e);
    delete c;
    return SWA_ERR_CUDA;
  }
  const StateLayout L = state_layout(cfg);
  char *base = static_cast<char *>(state_dev);
  const int64_t ps = cfg->page_size;
  c->np_full = cfg->size_full / ps;
  c->np_swa = cfg->size_swa / ps;
  c->mapping_len = cfg->size_full + ps + 1;
  c->counters = reinterpret_cast<int64_t *>(base + L.counters);
  c->mapping = reinterpret_cast<int64_t *>(base + L.mapping);
  int64_t *ev = reinterpret_cast<int64_t *>(base + L.ev);
  c->ev = swa::EvictScratch{ev, ev + cfg->max_batch, ev + 2 * cfg->max_batch, ev + 3 * cfg->max_batch};
  c->full = swa::PoolDev{reinterpret_cast<int64_t *>(base + L.ring_full),
                         reinterpret_cast<int64_t *>(base + L.staged_full),
                         c->counters + SWA_CTR_FULL_HEAD, c->counters + SWA_CTR_FULL_COUNT,
                         c->counters + SWA_CTR_FULL_STAGED, c->np_full};
  c->swa = swa::PoolDev{reinterpret_cast<int64_t *>(base + L.ring_swa),
                        reinterpret_cast<int64_t *>(base + L.staged_swa),
                        c->counters + SWA_CTR_SWA_HEAD, c->counters + SWA_CTR_SWA_COUNT,
                        c->counters + SWA_CTR_SWA_STAGED, c->np_swa};
  c->swa.ring_cost = c->ring_cost;
  c->swa.ring_slots = c->ring_slots;
  c->err_word = reinterpret_cast<int32_t *>(c->counters + SWA_CTR_ERROR);
  for (int l = 0; l < cfg->num_layers; ++l) swa::make_kv_tensor_maps(*c, l);
  c->h_count_full = c->np_full;
  c->h_count_swa = c->np_swa;
  e = swa::launch_init_state(*c, init_free_full, init_free_swa, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    g_create_err = std::string("init kernel: ") + cudaGetErrorString(e);
    delete c;
    return SWA_ERR_CUDA;
  }
  *out = c;
  return SWA_OK;
}

void swa_ctx_destroy(swa_ctx *ctx) { delete ctx; }

const char *swa_last_error(const swa_ctx *ctx) {
  return ctx ? ctx->err.c_str() : g_create_err.c_str();
}

swa_status swa_state_pointers(const swa_ctx *c, swa_state_view *o) {
  if (!c || !o) return SWA_ERR_INVALID;
  o->mapping = c->mapping;
  o->free_full = c->full.ring;
  o->staged_full = c->full.staged;
  o->free_swa = c->swa.ring;
  o->staged_swa = c->swa.staged;
  o->counters = c->counters;
  o->num_pages_full = c->np_full;
  o->num_pages_swa = c->np_swa;
  return SWA_OK;
}

int64_t swa_available_full(const swa_ctx *c) {
  if (!c || c->mirror_stale) return -1;
  return (c->h_count_full + c->h_staged_full) * c->cfg.page_size;
}
int64_t swa_available_swa(const swa_ctx *c) {
  if (!c || c->mirror_stale) return -1;
  if (c->ring_cost) return c->cfg.size_swa;   // rings are never exhausted
  return (c->h_count_swa + c->h_staged_swa) * c->cfg.page_size;
}
int64_t swa_available_size(const swa_ctx *c) {
  if (!c || c->mirror_stale) return -1;
  if (c->ring_cost) return swa_available_full(c);   // only the full pool can run out
  return std::min(swa_available_full(c), swa_available_swa(c));
}

swa_status swa_device_check(swa_ctx *c, swa_stream_t stream, int32_t *err) {
  SWA_NVTX("swa_device_check");
  if (!c) return SWA_ERR_INVALID;
  CUDA_TRY(c, cudaStreamSynchronize((cudaStream_t)stream));
  int32_t w = 0;
  CUDA_TRY(c, cudaMemcpy(&w, c->err_word, sizeof(w), cudaMemcpyDeviceToHost));
  CUDA_TRY(c, cudaMemset(c->err_word, 0, sizeof(int32_t)));
  if (err) *err = w;
  if (w) return fail(c, SWA_ERR_DEVICE_CHECK, "device check flagged error bits " + std::to_string(w));
  return SWA_OK;
}

swa_status swa_sync_counts(swa_ctx *c, swa_stream_t stream) {
  SWA_NVTX("swa_sync_counts");
  if (!c) return SWA_ERR_INVALID;
  CUDA_TRY(c, cudaStreamSynchronize((cudaStream_t)stream));
  int64_t h[8];
  CUDA_TRY(c, cudaMemcpy(h, c->counters, sizeof(h), cudaMemcpyDeviceToHost));
  c->h_count_full = h[SWA_CTR_FULL_COUNT];
  c->h_staged_full = h[SWA_CTR_FULL_STAGED];
  c->h_count_swa = h[SWA_CTR_SWA_COUNT];
  c->h_staged_swa = h[SWA_CTR_SWA_STAGED];
  c->mirror_stale = false;
  return SWA_OK;
}

// -------------------------------------------------------------- allocation ---
swa_status swa_alloc(swa_ctx *c, int64_t need, int64_t *out_full, int64_t *out_swa,
                     swa_stream_t stream) {
  SWA_NVTX("swa_alloc");
  if (!c || need < 0 || (need > 0 && !out_full)) return fail(c, SWA_ERR_INVALID, "bad alloc args");
  if (need % c->cfg.page_size) return fail(c, SWA_ERR_INVALID, "need_size is not page aligned");
  if (c->ring_cost) return fail(c, SWA_ERR_INVALID, "plain alloc has no request slot in ring mode");
  const int64_t n = need / c->cfg.page_size;
  if (n == 0) return SWA_OK;
  cudaStream_t s = (cudaStream_t)stream;
  bool okf = ensure_pages(c, true, n, s);
  bool oks = ensure_pages(c, false, n, s);
  if (!okf || !oks) return fail(c, SWA_ERR_NOMEM, "not enough free pages");
  CUDA_TRY(c, swa::launch_alloc_pages(*c, need, out_full, out_swa, s));
  c->h_count_full -= n;
  c->h_count_swa -= n;
  return SWA_OK;
}

static swa_status alloc_common(swa_ctx *c, int32_t bs, const int64_t *pre, const int64_t *seq,
                               const int64_t *last_loc, const int64_t *pre_h,
                               const int64_t *seq_h, int64_t *out_full, int64_t *out_swa,
                               int32_t *rt, int64_t rt_stride, const int64_t *req_idx,
                               swa_stream_t stream) {
  if (!c) return SWA_ERR_INVALID;
  if (bs < 0 || bs > c->cfg.max_batch) return fail(c, SWA_ERR_INVALID, "bs out of range");
  if (bs == 0) return SWA_OK;
  if (!seq || !seq_h) return fail(c, SWA_ERR_INVALID, "null lengths");
  if (!last_loc && !rt) return fail(c, SWA_ERR_INVALID, "need last_loc or req_to_token");
  if (rt && (!req_idx || rt_stride < 1)) return fail(c, SWA_ERR_INVALID, "req_to_token needs req_idx");
  if (c->ring_cost && !req_idx) return fail(c, SWA_ERR_INVALID, "ring mode needs req_idx");
  const int64_t ps = c->cfg.page_size;
  int64_t n_new = 0, n_tok = 0;
  for (int b = 0; b < bs; ++b) {
    const int64_t sq = seq_h[b], pr = pre_h ? pre_h[b] : seq_h[b] - 1;
    if (pr < 0 || sq < pr) return fail(c, SWA_ERR_INVALID, "need 0 <= prefix <= seq");
    if (rt && sq > rt_stride) return fail(c, SWA_ERR_INVALID, "seq exceeds req_to_token row");
    if (c->ring_cost && sq - pr + c->lookback > c->ring_cost)
      return fail(c, SWA_ERR_INVALID, "more new tokens than the ring holds beside the window");
    n_new += cdiv(sq, ps) - cdiv(pr, ps);
    n_tok += sq - pr;
  }
  if (n_tok > 0 && !out_full) return fail(c, SWA_ERR_INVALID, "null output");
  if (n_tok == 0) return SWA_OK;   // nothing to allocate
  cudaStream_t s = (cudaStream_t)stream;
  bool okf = ensure_pages(c, true, n_new, s);
  bool oks = c->ring_cost ? true : ensure_pages(c, false, n_new, s);
  if (!okf || !oks) return fail(c, SWA_ERR_NOMEM, "not enough free pages");
  CUDA_TRY(c, swa::launch_alloc_extend(*c, bs, pre, seq, last_loc, out_full, out_swa, rt,
                                        rt_stride, req_idx, 0, s));
  c->h_count_full -= n_new;
  if (!c->ring_cost) c->h_count_swa -= n_new;
  return SWA_OK;
}

swa_status swa_alloc_extend(swa_ctx *c, int32_t bs, const int64_t *prefix_lens,
                            const int64_t *seq_lens, const int64_t *last_loc,
                            const int64_t *prefix_lens_host, const int64_t *seq_lens_host,
                            int64_t *out_full, int64_t *out_swa, int32_t *req_to_token,
                            int64_t rt_stride, const int64_t *req_idx, swa_stream_t stream) {
  SWA_NVTX("swa_alloc_extend");
  if (c && bs > 0 && (!prefix_lens || !prefix_lens_host))
    return fail(c, SWA_ERR_INVALID, "null prefix lengths");
  return alloc_common(c, bs, prefix_lens, seq_lens, last_loc, prefix_lens_host, seq_lens_host,
                      out_full, out_swa, req_to_token, rt_stride, req_idx, stream);
}

swa_status swa_alloc_decode(swa_ctx *c, int32_t bs, const int64_t *seq_lens,
                            const int64_t *last_loc, const int64_t *seq_lens_host,
                            int64_t *out_full, int64_t *out_swa, int32_t *req_to_token,
                            int64_t rt_stride, const int64_t *req_idx, swa_stream_t stream) {
  SWA_NVTX("swa_alloc_decode");
  if (c && seq_lens_host)
    for (int b = 0; b < bs; ++b)
      if (seq_lens_host[b] < 1) return fail(c, SWA_ERR_INVALID, "decode seq_lens must be >= 1");
  return alloc_common(c, bs, nullptr, seq_lens, last_loc, nullptr, seq_lens_host, out_full,
                      out_swa, req_to_token, rt_stride, req_idx, stream);
}

swa_status swa_translate_for_kernel(swa_ctx *c, const int64_t *v2p, int64_t n_pages,
                                    const int64_t *virt, int64_t n, int32_t page_size,
                                    int32_t multiplier, int64_t *out, swa_stream_t stream) {
  SWA_NVTX("swa_translate_for_kernel");
  if (n < 0 || n_pages < 0 || page_size < 1 || multiplier < 1 ||
      (n > 0 && (!v2p || !virt || !out)))
    return fail(c, SWA_ERR_INVALID, "bad translate_for_kernel args");
  CUDA_TRY(c, swa::launch_translate_for_kernel(v2p, n_pages, virt, n, page_size, multiplier, out,
                                               c ? c->err_word : nullptr, c ? c->num_sms : 0,
                                               (cudaStream_t)stream));
  return SWA_OK;
}

swa_status swa_translate(swa_ctx *c, const int64_t *full_loc, int64_t n, int64_t *swa_loc,
                         swa_stream_t stream) {
  SWA_NVTX("swa_translate");
  if (!c || n < 0 || (n > 0 && (!full_loc || !swa_loc))) return fail(c, SWA_ERR_INVALID, "bad translate args");
  CUDA_TRY(c, swa::launch_translate(*c, full_loc, n, swa_loc, (cudaStream_t)stream));
  return SWA_OK;
}

// ----------------------------------------------------------------- release ---
swa_status swa_free(swa_ctx *c, const int64_t *full_idx, int64_t n, int64_t n_full_pages,
                    int64_t n_swa_pages, swa_stream_t stream) {
  SWA_NVTX("swa_free");
  if (!c || n < 0 || (n > 0 && !full_idx)) return fail(c, SWA_ERR_INVALID, "bad free args");
  if (n == 0) return SWA_OK;
  CUDA_TRY(c, swa::launch_release(*c, full_idx, n, true, n_full_pages, n_swa_pages,
                                  (cudaStream_t)stream));
  mirror_release(c, true, n_full_pages);
  if (!c->ring_cost) mirror_release(c, false, n_swa_pages);
  return SWA_OK;
}

swa_status swa_free_swa(swa_ctx *c, const int64_t *full_idx, int64_t n, int64_t n_swa_pages,
                        swa_stream_t stream) {
  SWA_NVTX("swa_free_swa");
  if (!c || n < 0 || (n > 0 && !full_idx)) return fail(c, SWA_ERR_INVALID, "bad free_swa args");
  if (n == 0) return SWA_OK;
  CUDA_TRY(c, swa::launch_release(*c, full_idx, n, false, -1, n_swa_pages, (cudaStream_t)stream));
  if (!c->ring_cost) mirror_release(c, false, n_swa_pages);
  return SWA_OK;
}

swa_status swa_evict_swa(swa_ctx *c, int32_t bs, const int32_t *rt, int64_t rt_stride,
                         const int64_t *req_idx, const int64_t *pre_lens, int64_t *evicted,
                         const int64_t *protected_lens, const int64_t *pre_h,
                         int64_t *evicted_h, const int64_t *protected_h, int32_t interval,
                         int32_t radix, swa_stream_t stream) {
  SWA_NVTX("swa_evict_swa");
  if (!c) return SWA_ERR_INVALID;
  if (bs < 0 || bs > c->cfg.max_batch) return fail(c, SWA_ERR_INVALID, "bs out of range");
  if (bs == 0) return SWA_OK;
  if (!rt || !req_idx || !pre_lens || !evicted || !pre_h || !evicted_h || interval < 0)
    return fail(c, SWA_ERR_INVALID, "bad evict args");
  const int64_t ps = c->cfg.page_size;
  const int64_t lb = radix ? std::max<int64_t>(c->lookback, ps) : c->lookback;
  int64_t total = 0;
  std::vector<int64_t> new_ev(evicted_h, evicted_h + bs);
  for (int b = 0; b < bs; ++b) {
    const int64_t ev = evicted_h[b];
    const int64_t bound = pre_h[b] - lb;
    if (interval > 0 && bound - ev < interval) continue;
    const int64_t nw = bound > 0 ? bound / ps * ps : 0;
    const int64_t prot = protected_h ? protected_h[b] : 0;
    const int64_t old = cdiv(std::max(ev, prot), ps) * ps;
    if (nw > old) {
      const int64_t n = (nw - old) / ps;
      if (nw > rt_stride) return fail(c, SWA_ERR_INVALID, "eviction range beyond req_to_token row");
      total += n;
      new_ev[b] = nw;
    }
  }
  // The host lengths decide exactly what the kernels would do (the lengths
  // travel with their device copies); a call that evicts nothing (most decode
  // steps between interval triggers) launches nothing.
  if (total > 0)
    CUDA_TRY(c, swa::launch_evict(*c, bs, rt, rt_stride, req_idx, pre_lens, evicted,
                                  protected_lens, interval, radix, (cudaStream_t)stream));
  if (!c->ring_cost) mirror_release(c, false, total);
  std::copy(new_ev.begin(), new_ev.end(), evicted_h);
  return SWA_OK;
}

// ------------------------------------------------------------------- store ---
swa_status swa_store_kv(swa_ctx *c, int32_t layer, const void *k, const void *v, int64_t n,
                        const int64_t *full_loc, const int64_t *swa_loc, float k_scale,
                        float v_scale, swa_stream_t stream) {
  SWA_NVTX("swa_store_kv");
  if (!c) return SWA_ERR_INVALID;
  if (layer < 0 || layer >= c->cfg.num_layers) return fail(c, SWA_ERR_INVALID, "layer out of range");
  if (n < 0 || (n > 0 && (!k || !v || !full_loc))) return fail(c, SWA_ERR_INVALID, "bad store args");
  if (c->cfg.kv_dtype == SWA_DTYPE_E4M3 && (!(k_scale > 0) || !(v_scale > 0)))
    return fail(c, SWA_ERR_INVALID, "fp8 scales must be > 0");
  CUDA_TRY(c, swa::launch_store(*c, layer, k, v, n, full_loc, swa_loc, k_scale, v_scale,
                                (cudaStream_t)stream));
  return SWA_OK;
}

// -------------------------------------------------------------------- plan ---
size_t swa_plan_bytes(const swa_ctx *c, int32_t bs, int32_t max_new) {
  if (!c || bs < 0) return 0;
  const size_t hdr = (((size_t)bs * 4 + 63) / 64) * 64 * sizeof(int32_t);
  return al256(hdr + (size_t)bs * swa::plan_max_pages(*c, max_new) * sizeof(int32_t));
}

swa_status swa_plan(swa_ctx *c, int32_t bs, const int32_t *rt, int64_t rt_stride,
                    const int64_t *req_idx, const int64_t *prefix_lens, const int64_t *seq_lens,
                    int32_t max_new, void *plan, size_t plan_bytes, swa_stream_t stream) {
  SWA_NVTX("swa_plan");
  if (!c) return SWA_ERR_INVALID;
  if (bs < 0 || bs > c->cfg.max_batch) return fail(c, SWA_ERR_INVALID, "bs out of range");
  if (bs == 0) return SWA_OK;
  if (!rt || !req_idx || !seq_lens || !plan || max_new < 1)
    return fail(c, SWA_ERR_INVALID, "bad plan args");
  if (plan_bytes < swa_plan_bytes(c, bs, max_new)) return fail(c, SWA_ERR_INVALID, "plan buffer too small");
  CUDA_TRY(c, swa::launch_plan(*c, bs, rt, rt_stride, req_idx, prefix_lens, seq_lens, max_new,
                               plan, (cudaStream_t)stream));
  return SWA_OK;
}

// --------------------------------------------------------------- attention ---
static bool use_mma(const swa_ctx *c, int layer) {
  return c->forced_path != 0 && swa::mma_decode_supported(*c, layer);
}
static bool use_tc(const swa_ctx *c, int layer) {
  return c->forced_path == -1 && swa::tc_extend_supported(*c, layer);
}

size_t swa_attn_decode_ws_bytes(const swa_ctx *c, int32_t layer, int32_t bs, int32_t max_seq_len) {
  if (!c || layer < 0 || layer >= c->cfg.num_layers || bs < 0 || max_seq_len < 1) return 0;
  if (use_mma(c, layer)) return swa::mma_decode_ws_bytes(*c, layer, bs, max_seq_len);
  return swa::simt_ws_bytes(*c, layer, bs, max_seq_len);
}

// Decode attention, optionally preceded by the store of the batch's new
// tokens: on the tensor-core path the attention launch stores them itself,
// elsewhere the store kernel runs first.
static swa_status attn_decode_impl(swa_ctx *c, int32_t layer, int32_t bs, const int32_t *rt,
                                   int64_t rt_stride, const int64_t *req_idx,
                                   const int64_t *seq_lens, int32_t max_seq_len, const void *plan,
                                   const void *q, const void *k_new, const void *v_new,
                                   const int64_t *full_loc, const int64_t *swa_loc,
                                   const float *sinks, float sm_scale, float k_scale,
                                   float v_scale, void *out, void *ws, size_t ws_bytes,
                                   swa_stream_t stream) {
  if (!c) return SWA_ERR_INVALID;
  if (layer < 0 || layer >= c->cfg.num_layers) return fail(c, SWA_ERR_INVALID, "layer out of range");
  if (bs < 0 || bs > c->cfg.max_batch) return fail(c, SWA_ERR_INVALID, "bs out of range");
  if (bs == 0) return SWA_OK;
  const swa::LayerInfo &L = c->layers[layer];
  if (!seq_lens || !q || !out || max_seq_len < 1 || (L.in_full && (!rt || !req_idx)) ||
      (!L.in_full && !plan))
    return fail(c, SWA_ERR_INVALID, "bad attention args");
  const bool store = k_new || v_new;
  if (store && (!k_new || !v_new || !full_loc)) return fail(c, SWA_ERR_INVALID, "bad store args");
  if (store && c->cfg.kv_dtype == SWA_DTYPE_E4M3 && (!(k_scale > 0) || !(v_scale > 0)))
    return fail(c, SWA_ERR_INVALID, "fp8 scales must be > 0");
  if (bs > 65535) return fail(c, SWA_ERR_INVALID, "bs > 65535");
  if (ws_bytes < swa_attn_decode_ws_bytes(c, layer, bs, max_seq_len) || !ws)
    return fail(c, SWA_ERR_INVALID, "split workspace too small");
  swa::AttnArgs a{};
  a.layer = layer;
  a.nq = bs;
  a.bs = bs;
  a.rt = rt;
  a.rt_stride = rt_stride;
  a.req_idx = req_idx;
  a.seq = seq_lens;
  a.max_seq_len = max_seq_len;
  a.max_new = 1;
  a.plan = plan_view(c, plan, bs, 1);
  a.q = q;
  a.sinks = sinks;
  a.scale = sm_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.out = out;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  cudaStream_t s = (cudaStream_t)stream;
  const bool mma = use_mma(c, layer);
  if (store && mma) {
    a.k_new = k_new;
    a.v_new = v_new;
    a.full_loc = full_loc;
    a.swa_loc = swa_loc;
  } else if (store) {
    CUDA_TRY(c, swa::launch_store(*c, layer, k_new, v_new, bs, full_loc, swa_loc, k_scale, v_scale, s));
  }
  if (mma) {
    c->last_path = 1;
    CUDA_TRY(c, swa::launch_attn_decode_mma(*c, a, s));
  } else {
    c->last_path = 0;
    CUDA_TRY(c, swa::launch_attn_simt(*c, a, s));
  }
  return SWA_OK;
}

swa_status swa_attn_decode(swa_ctx *c, int32_t layer, int32_t bs, const int32_t *rt,
                           int64_t rt_stride, const int64_t *req_idx, const int64_t *seq_lens,
                           int32_t max_seq_len, const void *plan, const void *q,
                           const float *sinks, float sm_scale, float k_scale, float v_scale,
                           void *out, void *ws, size_t ws_bytes, swa_stream_t stream) {
  SWA_NVTX("swa_attn_decode");
  return attn_decode_impl(c, layer, bs, rt, rt_stride, req_idx, seq_lens, max_seq_len, plan, q,
                          nullptr, nullptr, nullptr, nullptr, sinks, sm_scale, k_scale, v_scale,
                          out, ws, ws_bytes, stream);
}

swa_status swa_store_kv_attn_decode(swa_ctx *c, int32_t layer, int32_t bs, const int32_t *rt,
                                    int64_t rt_stride, const int64_t *req_idx,
                                    const int64_t *seq_lens, int32_t max_seq_len, const void *plan,
                                    const void *q, const void *k_new, const void *v_new,
                                    const int64_t *full_loc, const int64_t *swa_loc,
                                    const float *sinks, float sm_scale, float k_scale,
                                    float v_scale, void *out, void *ws, size_t ws_bytes,
                                    swa_stream_t stream) {
  SWA_NVTX("swa_store_kv_attn_decode");
  if (c && bs > 0 && (!k_new || !v_new || !full_loc)) return fail(c, SWA_ERR_INVALID, "bad store args");
  return attn_decode_impl(c, layer, bs, rt, rt_stride, req_idx, seq_lens, max_seq_len, plan, q,
                          k_new, v_new, full_loc, swa_loc, sinks, sm_scale, k_scale, v_scale, out,
                          ws, ws_bytes, stream);
}

size_t swa_attn_extend_ws_bytes(const swa_ctx *c, int32_t layer, int64_t n_tokens,
                                int32_t max_seq_len) {
  if (!c || layer < 0 || layer >= c->cfg.num_layers || n_tokens < 0 || max_seq_len < 1) return 0;
  if (use_tc(c, layer)) return swa::tc_extend_ws_bytes(*c, layer, n_tokens, max_seq_len);
  return swa::simt_ws_bytes(*c, layer, n_tokens, max_seq_len);
}

swa_status swa_attn_extend(swa_ctx *c, int32_t layer, int32_t bs, const int32_t *rt,
                           int64_t rt_stride, const int64_t *req_idx, const int64_t *prefix_lens,
                           const int64_t *seq_lens, const int64_t *qo_indptr, int64_t n_tokens,
                           int32_t max_new, int32_t max_seq_len, const void *plan, const void *q,
                           const float *sinks, float sm_scale, float k_scale, float v_scale,
                           void *out, void *ws, size_t ws_bytes, swa_stream_t stream) {
  SWA_NVTX("swa_attn_extend");
  if (!c) return SWA_ERR_INVALID;
  if (layer < 0 || layer >= c->cfg.num_layers) return fail(c, SWA_ERR_INVALID, "layer out of range");
  if (bs < 0 || bs > c->cfg.max_batch || n_tokens < 0) return fail(c, SWA_ERR_INVALID, "bs out of range");
  if (bs == 0 || n_tokens == 0) return SWA_OK;
  const swa::LayerInfo &L = c->layers[layer];
  if (!prefix_lens || !seq_lens || !qo_indptr || !q || !out || max_new < 1 || max_seq_len < 1 ||
      (L.in_full && (!rt || !req_idx)) || (!L.in_full && !plan))
    return fail(c, SWA_ERR_INVALID, "bad attention args");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(c, SWA_ERR_INVALID, "q and out must be 16-byte aligned");
  if (ws_bytes < swa_attn_extend_ws_bytes(c, layer, n_tokens, max_seq_len) || !ws)
    return fail(c, SWA_ERR_INVALID, "split workspace too small");
  const bool tc = use_tc(c, layer);
  if (!tc && n_tokens > 65535) return fail(c, SWA_ERR_INVALID, "n_tokens > 65535 on the generic path");
  swa::AttnArgs a{};
  a.layer = layer;
  a.nq = (int)n_tokens;
  a.bs = bs;
  a.rt = rt;
  a.rt_stride = rt_stride;
  a.req_idx = req_idx;
  a.pre = prefix_lens;
  a.seq = seq_lens;
  a.qo_indptr = qo_indptr;
  a.max_seq_len = max_seq_len;
  a.max_new = max_new;
  a.plan = plan_view(c, plan, bs, max_new);
  a.q = q;
  a.sinks = sinks;
  a.scale = sm_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.out = out;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  cudaStream_t s = (cudaStream_t)stream;
  if (tc) {
    c->last_path = 2;
    CUDA_TRY(c, swa::launch_attn_extend_tc(*c, a, s));
  } else {
    c->last_path = 0;
    CUDA_TRY(c, swa::launch_attn_simt(*c, a, s));
  }
  return SWA_OK;
}

int32_t swa_last_attn_path(const swa_ctx *c) { return c ? c->last_path : -1; }

swa_status swa_set_attn_path(swa_ctx *c, int32_t path) {
  if (!c) return SWA_ERR_INVALID;
  if (path < -1 || path > 1) return fail(c, SWA_ERR_INVALID, "path must be -1, 0 or 1");
  c->forced_path = path;
  return SWA_OK;
}

}  // extern "C"
