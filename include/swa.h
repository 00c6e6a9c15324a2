/*
 * libswa - hybrid sliding-window (SWA) two-pool KV cache and paged attention
 * for one NVIDIA GB300 (sm_103a).
 *
 * Method (source pages, cited by title and section):
 *   [SWA note]  "SWA in SGLang" design note (zdszero.github.io/swa.html)
 *   [Pools 15]  "SGLang source teardown (15): memory pools and allocators"
 *   [PR 34602]  SGLang PR #34602 summary, "unified pool MHA/SWA -> dense
 *               per-layer views" (prhub.com.cn)
 *
 * One token has two addresses: a slot in the FULL pool (its primary
 * address, kept while the request lives) and, through the mapping
 * full_to_swa[full_slot], a slot in the SWA pool that is returned once the
 * token slides out of every sliding window ([SWA note], "abstraction: one
 * token, two addresses").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Ownership: the caller allocates and owns every device buffer (KV pools,
 *   the state blob, req_to_token, q/out, plan and workspaces).  The library
 *   allocates no device memory; it keeps host-side mirrors of the free
 *   counts only.
 * - Asynchrony: every call enqueues work on `stream` and returns without
 *   synchronising, except swa_device_check() and swa_sync_counts().  Host
 *   copies of lengths are passed next to device copies so capacity checks
 *   need no device read ([Pools 15], "alloc_decode": the CPU copy of the
 *   lengths avoids an implicit sync).
 * - Errors: a non-SWA_OK status leaves device state and host mirrors
 *   untouched unless stated; swa_last_error() gives a message.  Kernels never
 *   trap: device-side checks (a read of mapping value 0 inside a window, a
 *   page count that disagrees with the host's) set an error word that
 *   swa_device_check() reads.
 * - Index types: slots, lengths, the mapping and free lists are int64;
 *   req_to_token is int32 ([Pools 15], ReqToTokenPool).  Slot 0 / page 0 of
 *   every pool is the padding sink and is never handed out.
 * - Layouts of one KV row (one token, one layer): [Hkv][D] elements.
 *   PER_LAYER: K and V of layer l are separate arrays of
 *   (pool_size + page_size) rows ([Pools 15], "second mapping", MHA pool).
 *   ENVELOPE: one byte buffer per pool of page envelopes
 *   [L0_K*ps | L0_V*ps | L1_K*ps | ...]; the row of slot t of pool-layer l is
 *   kernel_id(t) + (2l or 2l+1)*ps with kernel_id(t) = (t/ps)*(ps*2L) + t%ps
 *   ([PR 34602], "implementation", step 1).
 * - KV pools must be zero-filled when created, as the pages' pools are
 *   ([Pools 15], "second mapping": torch.zeros): the tensor-core kernels load
 *   whole pages, and rows of a page outside a query's key range must hold
 *   finite values (their softmax weight is zero).
 * - Streams: swa_stream_t is a cudaStream_t (0 = legacy default stream).
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *swa_stream_t;
typedef struct swa_ctx swa_ctx;

typedef enum swa_status {
  SWA_OK = 0,
  SWA_ERR_NOMEM = 1,        /* not enough free pages; nothing was changed      */
  SWA_ERR_INVALID = 2,      /* bad argument (null pointer, size, layer, ...)   */
  SWA_ERR_CONFIG = 3,       /* configuration rejected at create time           */
  SWA_ERR_CUDA = 4,         /* a CUDA runtime call failed                      */
  SWA_ERR_DEVICE_CHECK = 5  /* a kernel's own check failed (swa_device_check)  */
} swa_status;

enum swa_layer_kind {
  SWA_LAYER_FULL = 0,     /* keys 0..p, full pool                               */
  SWA_LAYER_SLIDING = 1,  /* keys max(0,p-window)..p, SWA pool; window excludes
                             the current token ([SWA note], "which models,
                             which layers": sliding_window - 1)               */
  SWA_LAYER_CHUNKED = 2   /* keys floor(p/C)*C..p with C = window, SWA pool    */
};

enum swa_dtype { SWA_DTYPE_F32 = 0, SWA_DTYPE_BF16 = 1, SWA_DTYPE_E4M3 = 2 };
enum swa_layout { SWA_LAYOUT_PER_LAYER = 0, SWA_LAYOUT_ENVELOPE = 1 };

/* Error-word bits set by device-side checks. */
enum swa_device_error {
  SWA_DEVERR_WINDOW_EVICTED = 1,  /* an attended key's SWA mapping was 0        */
  SWA_DEVERR_COUNT = 2,           /* freed page count differs from host count  */
  SWA_DEVERR_RANGE = 4,           /* slot / page / position out of range       */
  SWA_DEVERR_TIMEOUT = 8          /* a kernel gave up a bounded wait (its
                                     outputs for the launch are incomplete)    */
};

typedef struct swa_layer {
  int32_t kind;          /* enum swa_layer_kind                                 */
  int32_t window;        /* SLIDING: exclusive window Wx; CHUNKED: chunk C      */
  int32_t num_kv_heads;  /* Hkv of this layer (GQA: Hq % Hkv == 0)              */
  int32_t reserved;
  void *k;               /* PER_LAYER: K rows [pool_size + page_size][Hkv][D]   */
  void *v;               /* PER_LAYER: V rows, same shape; ENVELOPE: unused     */
} swa_layer;

typedef struct swa_config {
  int32_t num_layers;
  int32_t page_size;      /* ps >= 1                                              */
  int64_t size_full;      /* full pool token capacity, multiple of ps             */
  int64_t size_swa;       /* SWA pool token capacity, multiple of ps              */
  int32_t num_q_heads;    /* Hq                                                   */
  int32_t head_dim;       /* D (K and V), multiple of 8, <= 256                   */
  int32_t kv_dtype;       /* enum swa_dtype of the stored KV                      */
  int32_t layout;         /* enum swa_layout                                      */
  int32_t need_sort;      /* 1: stage released pages, sort-merge when short       */
  int32_t max_batch;      /* largest bs of any call                               */
  const swa_layer *layers;/* num_layers entries, copied at create                 */
  void *full_envelope;    /* ENVELOPE: full-pool byte buffer                      */
  int64_t full_envelope_bytes;
  void *swa_envelope;     /* ENVELOPE: SWA-pool byte buffer                       */
  int64_t swa_envelope_bytes;
  int32_t swa_ring_size;  /* > 0: per-request SWA rings (below); 0: paged SWA pool */
  int32_t ring_slots;     /* ring mode: request slots, req_idx in [0, ring_slots)   */
} swa_config;

/* Per-request SWA ring ([Pools 15], "why sliding windows can be accounted per
 * request"): instead of a paged SWA pool, every request slot owns one ring of
 * cost = ceil(swa_ring_size / page_size) * page_size SWA slots, and the SWA
 * pool holds exactly one ring per slot: size_swa must equal ring_slots * cost
 * (the pages' capacity rule).  Position t of the request in slot r lives at
 * SWA slot page_size + r * cost + t % cost (slots 0 .. page_size-1 stay the
 * padding page; the in-ring address is this library's reading, the pages do
 * not print it).  Consequences, all checked here:
 *   - alloc_extend / alloc_decode take SWA slots from the rings (req_idx is
 *     required) and still write mapping[full] = swa, so translate, the plan,
 *     the KV store and attention are unchanged; plain swa_alloc has no request
 *     slot and is SWA_ERR_INVALID;
 *   - only the full pool can run out (SWA_ERR_NOMEM); swa_available_swa is
 *     size_swa and swa_available_size is the full pool's;
 *   - swa_ring_size must be at least the largest SWA-layer lookback + 1, and a
 *     call may add at most cost - lookback tokens to a request (the ring holds
 *     the window plus every token stored before the attention that reads it),
 *     else SWA_ERR_INVALID;
 *   - swa_evict_swa and swa_free / swa_free_swa release no SWA pages: they
 *     zero the mapping entries of the tokens that left the window (so the
 *     device check on window reads keeps its meaning); the SWA page counts
 *     passed to them are ignored. */

/* Device pointers into the state blob, for inspection by tests. */
typedef struct swa_state_view {
  int64_t *mapping;        /* size_full + ps + 1 entries, last = -1           */
  int64_t *free_full;      /* ring of num_pages_full page ids                 */
  int64_t *staged_full;    /* num_pages_full                                  */
  int64_t *free_swa;       /* ring of num_pages_swa page ids                  */
  int64_t *staged_swa;
  int64_t *counters;       /* see SWA_CTR_* below                             */
  int64_t num_pages_full;
  int64_t num_pages_swa;
} swa_state_view;

enum swa_counter {
  SWA_CTR_FULL_HEAD = 0, SWA_CTR_FULL_COUNT = 1, SWA_CTR_FULL_STAGED = 2,
  SWA_CTR_SWA_HEAD = 3, SWA_CTR_SWA_COUNT = 4, SWA_CTR_SWA_STAGED = 5,
  SWA_CTR_ERROR = 6
};

/* ---------------------------------------------------------------- sizing --
 * Two-pool sizing ([SWA note], "how memory is split:
 * --swa-full-tokens-ratio"): cell = F*L_full + r*S*L_swa,
 * N_full = floor(M / cell), N_swa = r*N_full, both aligned down to a page.
 * F, S: KV bytes of one token in one full / SWA layer
 * (kv_heads * (head_dim + v_head_dim) * dtype_size).
 * Returns SWA_ERR_CONFIG when N_swa <= window + page_size (the SWA pool
 * cannot hold one request). Pure host function. */
swa_status swa_pool_sizes(int64_t mem_bytes, int64_t F, int64_t S,
                          int32_t L_full, int32_t L_swa, double r,
                          int32_t page_size, int32_t window,
                          int64_t *n_full, int64_t *n_swa);

/* Per-step decode allocation under speculative decoding ([Pools 15], "how
 * the sizes are set: from the memory budget to pool sizes").  algo:
 * SWA_SPEC_NONE (plain decode), SWA_SPEC_DRAFT (a draft tree of `topk`
 * branches, `steps` deep; has_draft_kv = 0 when drafts write no KV of their
 * own), SWA_SPEC_UNO (`draft_tokens` draft slots plus one clean root).
 * Outputs, in slots per request:
 *   alloc_len: one token without speculation; UNO: draft_tokens + 1; page
 *     size 1, one branch, or no draft KV: max(steps * topk, draft_tokens);
 *     otherwise every branch may start anywhere in a page and gets its own
 *     pages: max(ceil((page_size - 1 + steps) / page_size) * page_size * topk,
 *     draft_tokens);
 *   reserve: 2 * alloc_len (double buffer for the scheduler's committed
 *     length lagging the device);
 *   rt_extra: req_to_token columns beyond the context length: 4 +
 *     draft_tokens, raised with speculation on pages of more than one slot
 *     (or UNO) to reserve + page_size - 1.
 * A speculative step then takes alloc_len slots per request through
 * swa_alloc_extend (prefix = current length, seq = prefix + alloc_len).
 * Pure host function; SWA_ERR_INVALID for a null output, page_size < 1, or
 * UNO without draft_tokens (draft_tokens < 0 means "not given"). */
enum swa_spec_algo { SWA_SPEC_NONE = 0, SWA_SPEC_DRAFT = 1, SWA_SPEC_UNO = 2 };
swa_status swa_decode_alloc_sizes(int32_t algo, int32_t steps, int32_t topk,
                                  int32_t draft_tokens, int32_t has_draft_kv,
                                  int32_t page_size, int64_t *alloc_len,
                                  int64_t *reserve, int64_t *rt_extra);

/* ------------------------------------------------- radix prefix cache --
 * SWA component of the radix prefix cache ([SWA note], "prefix cache:
 * tombstones and the window hit rule").  A host-side tree over token ids that
 * holds full slots; a node whose SWA KV was released is a tombstone.
 *   - window: tokens that must hold live SWA KV before a match end (the SWA
 *     layers' largest lookback).  A match ends at the last page boundary e
 *     with min(e, window) live tokens before it (fewer than `window` only
 *     when the run of live tokens reaches the root);
 *   - full eviction deletes least recently used unlocked leaves; SWA eviction
 *     makes the least recently used unlocked live node a tombstone, or deletes
 *     it if it is a leaf (a leaf is never a tombstone; a tombstone left
 *     childless is deleted too);
 *   - a lock full-locks the path to the root and SWA-locks the nodes holding
 *     the last `window` tokens; it returns that span, which the unlock takes;
 *   - insert at request end: [0, swa_evicted) goes in as a tombstone prefix
 *     (only ahead of live tokens); a tombstone the request has SWA KV for is
 *     revived with the request's slots.
 * Readings (the page is silent): the tree works in whole pages (a trailing
 * partial page of a key is ignored: its slots stay the caller's); a match
 * splits the node it ends inside; every node a match passes, and every node
 * an insert passes or creates, takes the current time stamp in both LRU
 * lists; ties go to the older node; the request's slots duplicating cached
 * tokens are released, unless they are the node's own (a prefix the request
 * took from the tree).
 * The tree never touches the device.  Every call appends the slots whose KV
 * must go back to two lists, read (and cleared) with swa_radix_releases:
 * `full` slots go to swa_free (n_full / page_size full pages,
 * n_full_live / page_size of them still mapping SWA pages), `swa` slots to
 * swa_free_swa (n_swa / page_size SWA pages).  The pointers stay valid until
 * the next swa_radix_releases.  swa_radix_match writes the matched length e,
 * the slots of tokens [0, e) (slots_out: capacity n, or NULL) and the node
 * ending at e (0 = root).  SWA_ERR_INVALID for bad arguments, an unknown
 * node, an unlock that does not match a lock, or swa_evicted not a multiple
 * of page_size. */
typedef struct swa_radix swa_radix;
swa_status swa_radix_create(int32_t page_size, int32_t window, swa_radix **out);
void swa_radix_destroy(swa_radix *t);
swa_status swa_radix_match(swa_radix *t, const int32_t *tokens, int64_t n, int64_t *e,
                           int64_t *slots_out, int64_t *node);
swa_status swa_radix_insert(swa_radix *t, const int32_t *tokens, int64_t n,
                            const int64_t *slots, int64_t swa_evicted);
swa_status swa_radix_lock(swa_radix *t, int64_t node, int64_t *swa_span);
swa_status swa_radix_unlock(swa_radix *t, int64_t node, int64_t swa_span);
/* swa_only = 0: full eviction; 1: SWA eviction.  freed: tokens released. */
swa_status swa_radix_evict(swa_radix *t, int32_t swa_only, int64_t n_tokens, int64_t *freed);
swa_status swa_radix_releases(swa_radix *t, const int64_t **full, int64_t *n_full,
                              int64_t *n_full_live, const int64_t **swa, int64_t *n_swa);
swa_status swa_radix_sizes(const swa_radix *t, int64_t *cached_tokens, int64_t *live_tokens,
                           int64_t *nodes);

/* ------------------------------------------------------------- lifecycle --
 * swa_state_bytes: size of the device state blob (mapping, free-page rings,
 * staging lists, counters) for `cfg`; the caller allocates it (any
 * contents, 256-byte aligned).
 *
 * swa_ctx_create: validates `cfg`, copies it, and initialises the blob on
 * `stream`: mapping = 0 with the trailing -1 sentinel ([SWA note], "two
 * pools and the mapping"); free lists = 1..num_pages, or the caller's
 * permutation init_free_full / init_free_swa (device, num_pages entries,
 * nullable).  ENVELOPE checks ([PR 34602], "implementation", step 2):
 * row ids (num_pages+1)*2L*ps < 2^31 and a one-envelope tail pad; K and V
 * widths are equal by construction (one head_dim).  Returns SWA_ERR_CONFIG
 * for a rejected configuration, SWA_ERR_INVALID for null pointers. */
size_t swa_state_bytes(const swa_config *cfg);
swa_status swa_ctx_create(const swa_config *cfg, void *state_dev,
                          const int64_t *init_free_full,
                          const int64_t *init_free_swa, swa_stream_t stream,
                          swa_ctx **out);
void swa_ctx_destroy(swa_ctx *ctx);
/* Message of the last failure on ctx (or of swa_ctx_create when ctx is
 * NULL).  Valid until the next call on the same ctx. */
const char *swa_last_error(const swa_ctx *ctx);
swa_status swa_state_pointers(const swa_ctx *ctx, swa_state_view *out);

/* Host mirrors, in tokens ([SWA note]: available = min of the two pools;
 * [Pools 15]: staged pages count as free). */
int64_t swa_available_size(const swa_ctx *ctx);
int64_t swa_available_full(const swa_ctx *ctx);
int64_t swa_available_swa(const swa_ctx *ctx);

/* Synchronises `stream`, reads the error word into *err (0 = clean) and
 * clears it.  Returns SWA_ERR_DEVICE_CHECK when *err != 0. */
swa_status swa_device_check(swa_ctx *ctx, swa_stream_t stream, int32_t *err);
/* Synchronises `stream` and reloads the host mirrors from the device
 * counters (for callers that free without knowing page counts). */
swa_status swa_sync_counts(swa_ctx *ctx, swa_stream_t stream);

/* ------------------------------------------------------------ allocation --
 * All three allocate the same number of slots in both pools and then write
 * mapping[full] = swa ([SWA note], "two pools and the mapping").  Both
 * pools are checked before either is touched; on SWA_ERR_NOMEM nothing
 * changed except a need_sort merge, which the pages also run before the
 * check ([Pools 15], "expansion and shortage", "_release_page_ids").
 *
 * swa_alloc: need_size (multiple of ps) slots of whole pages, written to
 * out_full[need_size] (device), and out_swa when non-null. */
swa_status swa_alloc(swa_ctx *ctx, int64_t need_size, int64_t *out_full,
                     int64_t *out_swa, swa_stream_t stream);

/* swa_alloc_extend ([Pools 15], "alloc_extend"): request b of bs extends
 * from prefix_lens[b] to seq_lens[b] tokens.  Its slots follow its previous
 * slot last_loc[b] (-1 when the prefix is empty) inside the half-full page,
 * then fill new pages taken from the free list in request order.  Output
 * out_full[sum(seq - pre)] in request order (out_swa likewise, nullable).
 * last_loc may be NULL when req_to_token is given: it is then read as
 * req_to_token[req_idx[b], pre-1] (or -1).  When req_to_token is non-null
 * the new slots are also written to req_to_token[req_idx[b], pre..seq-1]
 * (row stride rt_stride int32 elements).  The *_host arrays are host copies
 * of prefix / seq lengths used for the page count. */
swa_status swa_alloc_extend(swa_ctx *ctx, int32_t bs,
                            const int64_t *prefix_lens, const int64_t *seq_lens,
                            const int64_t *last_loc,
                            const int64_t *prefix_lens_host,
                            const int64_t *seq_lens_host, int64_t *out_full,
                            int64_t *out_swa, int32_t *req_to_token,
                            int64_t rt_stride, const int64_t *req_idx,
                            swa_stream_t stream);

/* swa_alloc_decode ([Pools 15], "alloc_decode"): one token per request,
 * prefix = seq - 1: the slot is last_loc+1, or the first slot of a new page
 * when the token opens a page.  Same argument conventions as
 * swa_alloc_extend; out_full[bs]. */
swa_status swa_alloc_decode(swa_ctx *ctx, int32_t bs, const int64_t *seq_lens,
                            const int64_t *last_loc,
                            const int64_t *seq_lens_host, int64_t *out_full,
                            int64_t *out_swa, int32_t *req_to_token,
                            int64_t rt_stride, const int64_t *req_idx,
                            swa_stream_t stream);

/* Kernel-facing ids through a virtual-to-physical page table ([PR 34602],
 * multi_ended_allocator.py, "translate_kv_loc_for_kernel"): for each virtual
 * token id t, out = v2p[t / page_size] * (page_size * multiplier)
 * + t % page_size, clamped at 0 so a tombstone page (v2p = -1) reads the
 * page-0 sink.  multiplier = row blocks of one page (2 x the pool's layers in
 * the envelope layout; with v2p the identity this is the envelope's
 * kernel_id).  v2p: n_pages int64 on the device; virt, out: n int64 on the
 * device.  ctx may be NULL (then out-of-range virtual pages are only set to
 * 0); with a ctx they also set SWA_DEVERR_RANGE.  The swa_unified_* calls
 * below allocate a unified pool and fill its v2p tables. */
swa_status swa_translate_for_kernel(swa_ctx *ctx, const int64_t *v2p, int64_t n_pages,
                                    const int64_t *virt, int64_t n, int32_t page_size,
                                    int32_t multiplier, int64_t *out, swa_stream_t stream);

/* ------------------------------------------------- unified pool (two ends) --
 * FULL and SWA sub-pools sharing one virtual id space and one physical page
 * range, allocated from its two ends ([Pools 15], allocator-family table,
 * UnifiedSWATokenToKVPoolAllocator, and the note on UnifiedSWAAllocatorBase:
 * the shared ids replace the full->SWA table, the policy manages both
 * budgets; [PR 34602], multi_ended_allocator.py: virtual_to_physical).
 * Policy (this library's reading; the pages do not print one):
 *   - physical pages 1..num_pages (page 0 is the sink of both sides).  FULL
 *     takes pages upward from the low end, SWA downward from the high end;
 *     the pages between the two frontiers are free to either side;
 *   - a side reuses its released pages nearest its own end first (FULL the
 *     lowest, SWA the highest), then grows its frontier; after a release a
 *     frontier retracts over released pages of its side that border it;
 *   - virtual pages 1..num_pages (owned by the FULL side) come from a free
 *     ring, front first; released ids are prepended in ascending order;
 *   - every new virtual page gets one FULL and one SWA physical page, written
 *     to v2p_full[v] / v2p_swa[v]; a released SWA page leaves a tombstone -1
 *     (kernel ids clamp it to the sink).
 * A request's tokens get virtual slots v * page_size + t % page_size by the
 * same rule as swa_alloc_extend (the open page continues after last_loc; new
 * pages in request order); kernel-facing ids come from
 * swa_translate_for_kernel(NULL, v2p_full or v2p_swa, num_pages + 1, ...).
 * An allocation that needs n new pages fits iff n virtual pages are free and
 * max(0, n - released_full) + max(0, n - released_swa) <= the gap; otherwise
 * SWA_ERR_NOMEM and nothing changes.  Host mirror: exact after allocations;
 * a release leaves it stale (a retraction depends on which pages came back),
 * and the next allocation (or swa_unified_sync) reloads it with one stream
 * synchronisation; swa_unified_available_size returns -1 while it is stale.
 * State: caller-allocated device blob of swa_unified_state_bytes (256-byte
 * aligned); views of it through swa_unified_state_pointers. */
typedef struct swa_unified swa_unified;
typedef struct swa_unified_view {
  int64_t *v2p_full;          /* num_pages + 1 entries, -1 = none / tombstone  */
  int64_t *v2p_swa;
  uint32_t *released_full;    /* bitmap over page ids 0..num_pages             */
  uint32_t *released_swa;
  int64_t *virt_free;         /* ring of num_pages virtual page ids            */
  int64_t *counters;          /* SWA_UCTR_*                                    */
  int64_t num_pages;
} swa_unified_view;
enum swa_unified_counter {
  SWA_UCTR_LOW = 0,       /* highest page FULL has taken from the low end       */
  SWA_UCTR_HIGH = 1,      /* lowest page SWA has taken from the high end        */
  SWA_UCTR_REL_FULL = 2,  /* released FULL pages (set bits of released_full)    */
  SWA_UCTR_REL_SWA = 3,
  SWA_UCTR_VHEAD = 4,     /* front of the virtual-id ring                       */
  SWA_UCTR_VCOUNT = 5,    /* free virtual pages                                 */
  SWA_UCTR_ERROR = 6      /* device error word (int32, swa_device_error bits)   */
};
size_t swa_unified_state_bytes(int64_t num_pages, int32_t max_batch);
/* SWA_ERR_CONFIG when num_pages exceeds 1.7M or virtual slots would not fit
 * req_to_token's int32. */
swa_status swa_unified_create(int64_t num_pages, int32_t page_size, int32_t max_batch,
                              void *state_dev, swa_stream_t stream, swa_unified **out);
void swa_unified_destroy(swa_unified *u);
const char *swa_unified_last_error(const swa_unified *u);
swa_status swa_unified_state_pointers(const swa_unified *u, swa_unified_view *out);
int64_t swa_unified_available_size(const swa_unified *u);
swa_status swa_unified_sync(swa_unified *u, swa_stream_t stream);
swa_status swa_unified_device_check(swa_unified *u, swa_stream_t stream, int32_t *err);
/* Arguments as swa_alloc_extend; out_virt[sum(seq - pre)] receives virtual
 * slots, and req_to_token (when given) holds virtual slots. */
swa_status swa_unified_alloc_extend(swa_unified *u, int32_t bs, const int64_t *prefix_lens,
                                    const int64_t *seq_lens, const int64_t *last_loc,
                                    const int64_t *prefix_lens_host,
                                    const int64_t *seq_lens_host, int64_t *out_virt,
                                    int32_t *req_to_token, int64_t rt_stride,
                                    const int64_t *req_idx, swa_stream_t stream);
/* free_swa: releases the SWA page of each distinct virtual page of virt[n]
 * that still has one (tombstone); free: free_swa, then the FULL page and the
 * virtual page itself.  A virtual slot outside 1..num_pages pages sets
 * SWA_DEVERR_RANGE and is skipped. */
swa_status swa_unified_free_swa(swa_unified *u, const int64_t *virt, int64_t n,
                                swa_stream_t stream);
swa_status swa_unified_free(swa_unified *u, const int64_t *virt, int64_t n, swa_stream_t stream);
/* swa_evict_swa's ranges ([SWA note], "runtime") with window_excl as Wx, over
 * req_to_token holding virtual slots; each range's pages go through free_swa. */
swa_status swa_unified_evict_swa(swa_unified *u, int32_t bs, int32_t window_excl,
                                 const int32_t *req_to_token, int64_t rt_stride,
                                 const int64_t *req_idx, const int64_t *pre_lens,
                                 int64_t *evicted, const int64_t *protected_lens,
                                 const int64_t *pre_lens_host, int64_t *evicted_host,
                                 const int64_t *protected_host, int32_t interval, int32_t radix,
                                 swa_stream_t stream);

/* swa_translate: swa_loc[i] = full_to_swa[full_loc[i]], where full_loc -1
 * reads the trailing sentinel (-1) ([SWA note], "attention backend":
 * translate_loc_from_full_to_swa). */
swa_status swa_translate(swa_ctx *ctx, const int64_t *full_loc, int64_t n,
                         int64_t *swa_loc, swa_stream_t stream);

/* --------------------------------------------------------------- release --
 * swa_free ([SWA note], "two pools and the mapping"; [Pools 15], "free,
 * dedupe and free_group"): frees the full pages of full_idx[n] (page ids
 * deduplicated, in ascending order, prepended to the free list or staged
 * under need_sort), then runs swa_free_swa on the same indices.
 * n_full_pages / n_swa_pages: the caller's count of distinct pages each
 * side will get back (it updates the host mirrors without a sync; a kernel
 * that finds a different count sets SWA_DEVERR_COUNT).  Pass -1 when unknown
 * and call swa_sync_counts() before the next capacity query. */
swa_status swa_free(swa_ctx *ctx, const int64_t *full_idx, int64_t n,
                    int64_t n_full_pages, int64_t n_swa_pages,
                    swa_stream_t stream);
/* swa_free_swa: frees the SWA pages of those full_idx whose mapping is > 0,
 * then sets the mapping of every full_idx to 0, so calling it before
 * swa_free never frees a page twice. */
swa_status swa_free_swa(swa_ctx *ctx, const int64_t *full_idx, int64_t n,
                        int64_t n_swa_pages, swa_stream_t stream);

/* swa_evict_swa ([SWA note], "runtime: returning slid-out KV",
 * free_swa_out_of_window_slots): for each request b (in batch order),
 *   bound = pre_lens[b] - Wx            (radix == 0, chunk cache)
 *         = pre_lens[b] - max(Wx, ps)   (radix != 0)
 * with Wx the largest lookback of the model's SWA-pool layers (SLIDING: its
 * window; CHUNKED: C-1).  With interval > 0 (decode) the pass skips the
 * request unless bound - evicted[b] >= interval; interval == 0 always runs
 * (before a prefill chunk).  new = floor(bound/ps)*ps,
 * old = ceil(max(evicted[b], protected[b])/ps)*ps; if new > old the SWA
 * pages of req_to_token[req_idx[b], old:new] are freed (one page id per ps
 * positions, ascending within a request, later requests ahead of earlier
 * ones - the order of per-request frees), their mapping entries set to 0,
 * and evicted[b] = new.  Device arrays drive the kernel; the *_host arrays
 * (same values) drive the host mirror, and evicted_host is updated too.
 * When the host arrays show that no request frees a page, no kernel is
 * launched.  protected may be NULL (all 0). */
swa_status swa_evict_swa(swa_ctx *ctx, int32_t bs, const int32_t *req_to_token,
                         int64_t rt_stride, const int64_t *req_idx,
                         const int64_t *pre_lens, int64_t *evicted,
                         const int64_t *protected_lens,
                         const int64_t *pre_lens_host, int64_t *evicted_host,
                         const int64_t *protected_host, int32_t interval,
                         int32_t radix, swa_stream_t stream);

/* ------------------------------------------------------------------ store --
 * swa_store_kv ([Pools 15], "who writes into the pages", KVWriteLoc):
 * k, v: [n][Hkv][D] rows of the new tokens of `layer` (f32 for an F32 pool,
 * bf16 otherwise).  A FULL layer writes row i at full_loc[i]; other layers
 * at swa_loc[i] (pre-translated once per batch; when NULL the mapping is
 * read here).  E4M3 pools store round-to-nearest-even, saturating
 * e4m3(x / scale) bytes ([Pools 15]: FP8 is kept as uint8). */
swa_status swa_store_kv(swa_ctx *ctx, int32_t layer, const void *k,
                        const void *v, int64_t n, const int64_t *full_loc,
                        const int64_t *swa_loc, float k_scale, float v_scale,
                        swa_stream_t stream);

/* ------------------------------------------------------------------- plan --
 * Per-batch translation done once and shared by every SWA-pool layer
 * ([SWA note], "attention backend: translate once"): for request b it
 * lists the SWA pages holding positions lo_b..hi_b, with
 *   decode:  hi_b = seq_lens[b] - 1,  lo_b = max(0, hi_b - Wx)
 *   extend:  hi_b = seq_lens[b] - 1,  lo_b = max(0, prefix_lens[b] - Wx)
 * (Wx as in swa_evict_swa).  A position whose SWA mapping is 0 sets
 * SWA_DEVERR_WINDOW_EVICTED.  `max_new` bounds seq - prefix over the batch
 * (1 for decode).  swa_plan_bytes gives the workspace size. */
size_t swa_plan_bytes(const swa_ctx *ctx, int32_t bs, int32_t max_new);
swa_status swa_plan(swa_ctx *ctx, int32_t bs, const int32_t *req_to_token,
                    int64_t rt_stride, const int64_t *req_idx,
                    const int64_t *prefix_lens /* NULL = decode */,
                    const int64_t *seq_lens, int32_t max_new, void *plan,
                    size_t plan_bytes, swa_stream_t stream);

/* ------------------------------------------------------------- attention --
 * For a query at position p, query head h, KV head h / (Hq / Hkv), key set
 * J (by layer kind, above), scale c and sink logit sigma_h ([SWA note],
 * "design": learnable sink):
 *   o_h = sum_j e^{c q.k_j - m} v_j / (e^{sigma_h - m} + sum_j e^{c q.k_j - m})
 * sinks: [Hq] float logits, or NULL for no sink.  q, out: [n][Hq][D], f32
 * for an F32 pool, bf16 otherwise.  E4M3 K/V are multiplied by k_scale /
 * v_scale after decoding.  Keys of FULL layers are read through
 * req_to_token, keys of SWA-pool layers through `plan` (built for the same
 * batch).  Long key ranges are split across CTAs and merged in the same
 * launch; `ws` is the split workspace (size from *_ws_bytes) and must be
 * zero-filled before its first use (the kernels leave it reusable).  Its
 * layout is [256 B counters][tickets][partials] with a ticket block of one
 * size per context for batches up to max_batch, so decode calls of any
 * layers may share one workspace sized for the largest of them; a generic-
 * path extend call with more query tokens than max_batch needs its own.
 *
 * swa_attn_decode: one query per request at p = seq_lens[b] - 1 (its KV
 * already stored). max_seq_len bounds seq_lens (host; sizes the grid).  On
 * the tensor-core path the launch is a programmatic dependent of the kernel
 * before it on the stream: it may be scheduled while that kernel finishes,
 * but reads nothing until that kernel has completed, so stream order and
 * every input the previous kernel wrote are respected as for a plain launch. */
size_t swa_attn_decode_ws_bytes(const swa_ctx *ctx, int32_t layer, int32_t bs,
                                int32_t max_seq_len);
swa_status swa_attn_decode(swa_ctx *ctx, int32_t layer, int32_t bs,
                           const int32_t *req_to_token, int64_t rt_stride,
                           const int64_t *req_idx, const int64_t *seq_lens,
                           int32_t max_seq_len, const void *plan, const void *q,
                           const float *sinks, float sm_scale, float k_scale,
                           float v_scale, void *out, void *ws, size_t ws_bytes,
                           swa_stream_t stream);

/* swa_store_kv_attn_decode: swa_store_kv of the batch's new tokens followed
 * by swa_attn_decode on the same layer, as one call ([Pools 15], "who writes
 * into the pages": the decode step stores each layer's new K/V, then that
 * layer attends over it).  k_new, v_new: [bs][Hkv][D] rows, laid out and
 * typed as for swa_store_kv (bf16 for bf16 and E4M3 pools, f32 for an F32
 * pool); row b is request b's token at p = seq_lens[b] - 1, stored at
 * full_loc[b] (full layers) or swa_loc[b] (SWA-pool layers; NULL =
 * mapping[full_loc[b]]) - the slots swa_alloc_decode returned, which
 * req_to_token / plan must map p to.  k_scale / v_scale serve both the E4M3
 * encoding of the store and the decoding in attention.  Where the
 * tensor-core decode kernel runs, one launch does both: the CTA whose key
 * range ends at p writes that token's row of its KV head, then loads it with
 * its other keys; on the other attention paths the store kernel runs first.
 * Pools and outputs are identical to the two calls in sequence.  Errors: as
 * the two calls (an out-of-range slot sets SWA_DEVERR_RANGE and is not
 * written). */
swa_status swa_store_kv_attn_decode(swa_ctx *ctx, int32_t layer, int32_t bs,
                                    const int32_t *req_to_token,
                                    int64_t rt_stride, const int64_t *req_idx,
                                    const int64_t *seq_lens,
                                    int32_t max_seq_len, const void *plan,
                                    const void *q, const void *k_new,
                                    const void *v_new, const int64_t *full_loc,
                                    const int64_t *swa_loc, const float *sinks,
                                    float sm_scale, float k_scale,
                                    float v_scale, void *out, void *ws,
                                    size_t ws_bytes, swa_stream_t stream);

/* swa_attn_decode_noalloc: swa_attn_decode for callers that cannot allocate
 * device memory - engines that give all of HBM to their KV pools at start-up
 * and allow no later allocation, plug-ins whose host framework exposes no
 * allocator, and paths where a cudaMalloc (which can synchronise the device)
 * is not acceptable.  The source pages have no counterpart; it exists for
 * those callers.  Arguments are swa_attn_decode's without ws / ws_bytes: the
 * split-KV scratch is a fixed 32 MiB array inside the library
 * (swa_attn_decode_noalloc_max_bytes()), which every GPU that loads the
 * library holds until the process exits.  A batch whose scratch
 * (swa_attn_decode_ws_bytes) exceeds it is rejected with SWA_ERR_INVALID and
 * a message.  The call allocates nothing: it looks up the array's device
 * address (a host-side query, on every call, so no address outlives a
 * cudaDeviceReset), clears the array's counters and merge tickets
 * (cudaMemsetAsync on `stream`; the partial results are not cleared - the
 * kernels write each one before reading it) and runs the same kernels as
 * swa_attn_decode.  The first call on a device loads the array onto that
 * device, so make that first call before any stream capture.  All calls on a
 * device share the array and it keeps the last call's contents; calls that
 * overlap on the GPU (e.g. on different streams) race on it. */
size_t swa_attn_decode_noalloc_max_bytes(void);
swa_status swa_attn_decode_noalloc(swa_ctx *ctx, int32_t layer, int32_t bs,
                                   const int32_t *req_to_token,
                                   int64_t rt_stride, const int64_t *req_idx,
                                   const int64_t *seq_lens, int32_t max_seq_len,
                                   const void *plan, const void *q,
                                   const float *sinks, float sm_scale,
                                   float k_scale, float v_scale, void *out,
                                   swa_stream_t stream);

/* swa_attn_extend: chunked-prefill queries.  Request b owns query rows
 * qo_indptr[b]..qo_indptr[b+1]-1 (device, bs+1 entries), at positions
 * prefix_lens[b] .. seq_lens[b]-1, causal.  n_tokens = qo_indptr[bs] and
 * max_new >= max(seq - prefix) are host values.  q and out are device
 * [n_tokens][num_q_heads][head_dim] arrays (f32 for an F32 pool, bf16
 * otherwise), both 16-byte aligned (SWA_ERR_INVALID otherwise).  The tcgen05
 * kernel serves bf16 pools with head_dim 64 or 128 and E4M3 pools with
 * head_dim 128, any query-per-KV-head group up to 128 and page sizes 16..64;
 * other configurations run the generic kernel, which takes at most 65535
 * tokens per call. */
size_t swa_attn_extend_ws_bytes(const swa_ctx *ctx, int32_t layer,
                                int64_t n_tokens, int32_t max_seq_len);
swa_status swa_attn_extend(swa_ctx *ctx, int32_t layer, int32_t bs,
                           const int32_t *req_to_token, int64_t rt_stride,
                           const int64_t *req_idx, const int64_t *prefix_lens,
                           const int64_t *seq_lens, const int64_t *qo_indptr,
                           int64_t n_tokens, int32_t max_new,
                           int32_t max_seq_len, const void *plan, const void *q,
                           const float *sinks, float sm_scale, float k_scale,
                           float v_scale, void *out, void *ws, size_t ws_bytes,
                           swa_stream_t stream);

/* Which kernel family the last attention call on ctx launched
 * (0 = generic CUDA-core kernel, 1 = tensor-core decode fed by cp.async,
 * 2 = tcgen05 extend), for tests and profiling. */
int32_t swa_last_attn_path(const swa_ctx *ctx);
/* Restricts the kernel family attention calls on ctx may take: -1 = best
 * available (default: cp.async tensor-core decode, tcgen05 extend), 0 =
 * generic CUDA-core kernel only, 1 = cp.async tensor-core decode and no
 * tcgen05 extend.  Any other value is SWA_ERR_INVALID.  For tests and
 * profiling. */
swa_status swa_set_attn_path(swa_ctx *ctx, int32_t path);

#ifdef __cplusplus
}
#endif
#endif /* SWA_H */
