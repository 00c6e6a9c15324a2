"""Thin ctypes binding of libswa (include/swa.h).

Argument marshalling only: every function has the C entry point's name and
calls it; device buffers are torch CUDA tensors (passed by data pointer),
host length arrays are numpy int64 arrays.  torch supplies device memory and
the current CUDA stream.  There is no fallback: if libswa.so is missing or
fails to load, the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libswa.so")

SWA_OK, SWA_ERR_NOMEM, SWA_ERR_INVALID, SWA_ERR_CONFIG, SWA_ERR_CUDA, SWA_ERR_DEVICE_CHECK = range(6)
LAYER_FULL, LAYER_SLIDING, LAYER_CHUNKED = 0, 1, 2
DTYPE_F32, DTYPE_BF16, DTYPE_E4M3 = 0, 1, 2
LAYOUT_PER_LAYER, LAYOUT_ENVELOPE = 0, 1
CTR_FULL_HEAD, CTR_FULL_COUNT, CTR_FULL_STAGED, CTR_SWA_HEAD, CTR_SWA_COUNT, CTR_SWA_STAGED, CTR_ERROR = range(7)
SWA_DEVERR_WINDOW_EVICTED, SWA_DEVERR_COUNT, SWA_DEVERR_RANGE, SWA_DEVERR_TIMEOUT = 1, 2, 4, 8

_STORE_TORCH = {DTYPE_F32: torch.float32, DTYPE_BF16: torch.bfloat16, DTYPE_E4M3: torch.uint8}


class SwaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libswa status {status}: {msg}")
        self.status = status


class SwaNoMem(SwaError):
    pass


class swa_layer(C.Structure):
    _fields_ = [("kind", C.c_int32), ("window", C.c_int32), ("num_kv_heads", C.c_int32),
                ("reserved", C.c_int32), ("k", C.c_void_p), ("v", C.c_void_p)]


class swa_config(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("page_size", C.c_int32),
                ("size_full", C.c_int64), ("size_swa", C.c_int64),
                ("num_q_heads", C.c_int32), ("head_dim", C.c_int32),
                ("kv_dtype", C.c_int32), ("layout", C.c_int32),
                ("need_sort", C.c_int32), ("max_batch", C.c_int32),
                ("layers", C.POINTER(swa_layer)),
                ("full_envelope", C.c_void_p), ("full_envelope_bytes", C.c_int64),
                ("swa_envelope", C.c_void_p), ("swa_envelope_bytes", C.c_int64),
                ("swa_ring_size", C.c_int32), ("ring_slots", C.c_int32)]


class swa_state_view(C.Structure):
    _fields_ = [("mapping", C.c_void_p), ("free_full", C.c_void_p), ("staged_full", C.c_void_p),
                ("free_swa", C.c_void_p), ("staged_swa", C.c_void_p), ("counters", C.c_void_p),
                ("num_pages_full", C.c_int64), ("num_pages_swa", C.c_int64)]


P = C.c_void_p
I32, I64, F32, SZ = C.c_int32, C.c_int64, C.c_float, C.c_size_t

# name -> (restype, argtypes): mirrors include/swa.h and include/swa_synth.h
SIGNATURES = {
    "swa_pool_sizes": (I32, [I64, I64, I64, I32, I32, C.c_double, I32, I32, P, P]),
    "swa_decode_alloc_sizes": (I32, [I32, I32, I32, I32, I32, I32, P, P, P]),
    "swa_translate_for_kernel": (I32, [P, P, I64, P, I64, I32, I32, P, P]),
    "swa_radix_create": (I32, [I32, I32, P]),
    "swa_radix_destroy": (None, [P]),
    "swa_radix_match": (I32, [P, P, I64, P, P, P]),
    "swa_radix_insert": (I32, [P, P, I64, P, I64]),
    "swa_radix_lock": (I32, [P, I64, P]),
    "swa_radix_unlock": (I32, [P, I64, I64]),
    "swa_radix_evict": (I32, [P, I32, I64, P]),
    "swa_radix_releases": (I32, [P, P, P, P, P, P]),
    "swa_radix_sizes": (I32, [P, P, P, P]),
    "swa_state_bytes": (SZ, [P]),
    "swa_ctx_create": (I32, [P, P, P, P, P, P]),
    "swa_ctx_destroy": (None, [P]),
    "swa_last_error": (C.c_char_p, [P]),
    "swa_state_pointers": (I32, [P, P]),
    "swa_available_size": (I64, [P]),
    "swa_available_full": (I64, [P]),
    "swa_available_swa": (I64, [P]),
    "swa_device_check": (I32, [P, P, P]),
    "swa_sync_counts": (I32, [P, P]),
    "swa_alloc": (I32, [P, I64, P, P, P]),
    "swa_alloc_extend": (I32, [P, I32, P, P, P, P, P, P, P, P, I64, P, P]),
    "swa_alloc_decode": (I32, [P, I32, P, P, P, P, P, P, I64, P, P]),
    "swa_translate": (I32, [P, P, I64, P, P]),
    "swa_free": (I32, [P, P, I64, I64, I64, P]),
    "swa_free_swa": (I32, [P, P, I64, I64, P]),
    "swa_evict_swa": (I32, [P, I32, P, I64, P, P, P, P, P, P, P, I32, I32, P]),
    "swa_store_kv": (I32, [P, I32, P, P, I64, P, P, F32, F32, P]),
    "swa_plan_bytes": (SZ, [P, I32, I32]),
    "swa_plan": (I32, [P, I32, P, I64, P, P, P, I32, P, SZ, P]),
    "swa_attn_decode_ws_bytes": (SZ, [P, I32, I32, I32]),
    "swa_attn_decode": (I32, [P, I32, I32, P, I64, P, P, I32, P, P, P, F32, F32, F32, P, P, SZ, P]),
    "swa_store_kv_attn_decode": (I32, [P, I32, I32, P, I64, P, P, I32, P, P, P, P, P, P, P, F32,
                                        F32, F32, P, P, SZ, P]),
    "swa_attn_decode_noalloc_max_bytes": (SZ, []),
    "swa_attn_decode_noalloc": (I32, [P, I32, I32, P, I64, P, P, I32, P, P, P, F32, F32, F32, P,
                                      P]),
    "swa_attn_extend_ws_bytes": (SZ, [P, I32, I64, I32]),
    "swa_attn_extend": (I32, [P, I32, I32, P, I64, P, P, P, P, I64, I32, I32, P, P, P, F32, F32,
                              F32, P, P, SZ, P]),
    "swa_last_attn_path": (I32, [P]),
    "swa_set_attn_path": (I32, [P, I32]),
    "swa_synth_tokens": (I32, [C.c_uint64, I32, I32, P, P, I64, I32, I32, I32, P, P]),
    "swa_unified_state_bytes": (SZ, [I64, I32]),
    "swa_unified_create": (I32, [I64, I32, I32, P, P, P]),
    "swa_unified_destroy": (None, [P]),
    "swa_unified_last_error": (C.c_char_p, [P]),
    "swa_unified_state_pointers": (I32, [P, P]),
    "swa_unified_available_size": (I64, [P]),
    "swa_unified_sync": (I32, [P, P]),
    "swa_unified_device_check": (I32, [P, P, P]),
    "swa_unified_alloc_extend": (I32, [P, I32, P, P, P, P, P, P, P, I64, P, P]),
    "swa_unified_free_swa": (I32, [P, P, I64, P]),
    "swa_unified_free": (I32, [P, P, I64, P]),
    "swa_unified_evict_swa": (I32, [P, I32, I32, P, I64, P, P, P, P, P, P, P, I32, I32, P]),
}

_lib = None


def lib():
    """Load libswa.so (raises if it is missing or lacks a symbol)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "python -m hybrid_sliding_window_gb300.build")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        assert t.is_cuda, "device buffer expected"
        assert t.is_contiguous()
        return t.data_ptr()
    return t


def _host(a):
    """Host int64 array -> (keepalive, pointer)."""
    if a is None:
        return None, None
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return arr, arr.ctypes.data_as(C.c_void_p)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(status, ctx_handle=None):
    if status != SWA_OK:
        msg = lib().swa_last_error(ctx_handle)
        msg = msg.decode() if msg else ""
        cls = SwaNoMem if status == SWA_ERR_NOMEM else SwaError
        raise cls(status, msg)


class SwaCtx:
    """Owns a libswa context, its device state blob and the config copy."""

    def __init__(self, layers, page_size, size_full, size_swa, num_q_heads, head_dim,
                 kv_dtype, layout=LAYOUT_PER_LAYER, need_sort=False, max_batch=256,
                 full_envelope=None, swa_envelope=None, init_free_full=None,
                 init_free_swa=None, device="cuda", stream=None, ring_size=0, ring_slots=0):
        """``layers``: list of dicts with keys kind, window, num_kv_heads and,
        for the per-layer layout, k / v tensors.  ``ring_size`` > 0 selects
        per-request SWA rings (``size_swa`` = ``ring_slots`` x ring cost)."""
        arr = (swa_layer * len(layers))()
        for i, d in enumerate(layers):
            arr[i].kind = d["kind"]
            arr[i].window = d.get("window", 0)
            arr[i].num_kv_heads = d["num_kv_heads"]
            arr[i].k = _ptr(d.get("k"))
            arr[i].v = _ptr(d.get("v"))
        cfg = swa_config()
        cfg.num_layers = len(layers)
        cfg.page_size = page_size
        cfg.size_full = size_full
        cfg.size_swa = size_swa
        cfg.num_q_heads = num_q_heads
        cfg.head_dim = head_dim
        cfg.kv_dtype = kv_dtype
        cfg.layout = layout
        cfg.need_sort = 1 if need_sort else 0
        cfg.max_batch = max_batch
        cfg.layers = C.cast(arr, C.POINTER(swa_layer))
        cfg.full_envelope = _ptr(full_envelope)
        cfg.full_envelope_bytes = full_envelope.numel() if full_envelope is not None else 0
        cfg.swa_envelope = _ptr(swa_envelope)
        cfg.swa_envelope_bytes = swa_envelope.numel() if swa_envelope is not None else 0
        cfg.swa_ring_size = ring_size
        cfg.ring_slots = ring_slots
        self.cfg = cfg
        self._layers_arr = arr
        self.layers = layers
        self.full_envelope = full_envelope
        self.swa_envelope = swa_envelope
        nbytes = lib().swa_state_bytes(C.byref(cfg))
        if nbytes == 0:
            raise SwaError(SWA_ERR_INVALID, "swa_state_bytes rejected the config")
        self.state = torch.empty(nbytes, dtype=torch.uint8, device=device)
        handle = C.c_void_p()
        st = lib().swa_ctx_create(C.byref(cfg), _ptr(self.state), _ptr(init_free_full),
                                  _ptr(init_free_swa), _stream(stream), C.byref(handle))
        _check(st, None)
        self.handle = handle
        view = swa_state_view()
        _check(lib().swa_state_pointers(handle, C.byref(view)), handle)
        self.view = view

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.swa_ctx_destroy(h)
            self.handle = None

    # -- inspection helpers (device -> host copies, for tests) ------------------
    def _dev_tensor(self, ptr, n):
        base = self.state.data_ptr()
        off = (ptr - base) // 8
        return self.state.view(torch.int64)[off:off + n]

    def mapping(self):
        return self._dev_tensor(self.view.mapping, self.cfg.size_full + self.cfg.page_size + 1)

    def counters(self):
        return self._dev_tensor(self.view.counters, 8)

    def free_list(self, full: bool):
        """Free pages in order (front first) and the staged pages."""
        ctr = self.counters().cpu().numpy()
        if full:
            ring = self._dev_tensor(self.view.free_full, self.view.num_pages_full).cpu().numpy()
            stg = self._dev_tensor(self.view.staged_full, self.view.num_pages_full).cpu().numpy()
            head, cnt, ns = ctr[CTR_FULL_HEAD], ctr[CTR_FULL_COUNT], ctr[CTR_FULL_STAGED]
        else:
            ring = self._dev_tensor(self.view.free_swa, self.view.num_pages_swa).cpu().numpy()
            stg = self._dev_tensor(self.view.staged_swa, self.view.num_pages_swa).cpu().numpy()
            head, cnt, ns = ctr[CTR_SWA_HEAD], ctr[CTR_SWA_COUNT], ctr[CTR_SWA_STAGED]
        cap = len(ring)
        idx = (head + np.arange(cnt)) % cap if cap else np.zeros(0, np.int64)
        return ring[idx].tolist(), stg[:ns].tolist()


# ------------------------------------------------------------- entry points ---
def swa_pool_sizes(mem_bytes, F, S, L_full, L_swa, r, page_size, window):
    nf, ns = C.c_int64(), C.c_int64()
    st = lib().swa_pool_sizes(mem_bytes, F, S, L_full, L_swa, r, page_size, window,
                              C.byref(nf), C.byref(ns))
    _check(st, None)
    return nf.value, ns.value


def swa_decode_alloc_sizes(algo, steps, topk, draft_tokens, has_draft_kv, page_size):
    """(alloc_len, reserve, rt_extra) per request per decode step;
    draft_tokens None means "not given"."""
    a, r, e = C.c_int64(), C.c_int64(), C.c_int64()
    st = lib().swa_decode_alloc_sizes(algo, steps, topk, -1 if draft_tokens is None else draft_tokens,
                                      1 if has_draft_kv else 0, page_size, C.byref(a), C.byref(r),
                                      C.byref(e))
    _check(st, None)
    return a.value, r.value, e.value


def swa_translate_for_kernel(v2p, virt, page_size, multiplier, out=None, ctx=None, stream=None):
    """Kernel-facing ids of virtual token ids through the page table v2p."""
    if out is None:
        out = torch.empty_like(virt)
    st = lib().swa_translate_for_kernel(ctx.handle if ctx is not None else None, _ptr(v2p),
                                        v2p.numel(), _ptr(virt), virt.numel(), page_size,
                                        multiplier, _ptr(out), _stream(stream))
    _check(st, ctx.handle if ctx is not None else None)
    return out


class RadixSWA:
    """The native SWA radix tree (include/swa.h, "radix prefix cache").
    Host only; releases come back as numpy arrays (see ``apply_releases``)."""

    def __init__(self, page_size, window):
        h = C.c_void_p()
        _check(lib().swa_radix_create(page_size, window, C.byref(h)), None)
        self.h = h
        self.ps = page_size

    def __del__(self):
        h = getattr(self, "h", None)
        if h is not None and _lib is not None:
            _lib.swa_radix_destroy(h)
            self.h = None

    def match(self, tokens, as_numpy=False):
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(max(len(t), 1), np.int64)
        e, node = C.c_int64(), C.c_int64()
        _check(lib().swa_radix_match(self.h, t.ctypes.data, len(t), C.byref(e),
                                     out.ctypes.data, C.byref(node)), None)
        slots = out[:e.value]
        return e.value, (slots if as_numpy else slots.tolist()), node.value

    def insert(self, tokens, slots, swa_evicted):
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        s = np.ascontiguousarray(slots, dtype=np.int64)
        _check(lib().swa_radix_insert(self.h, t.ctypes.data, min(len(t), len(s)), s.ctypes.data,
                                      swa_evicted), None)

    def lock(self, node):
        span = C.c_int64()
        _check(lib().swa_radix_lock(self.h, node, C.byref(span)), None)
        return span.value

    def unlock(self, node, span):
        _check(lib().swa_radix_unlock(self.h, node, span), None)

    def evict(self, n_tokens, swa_only=False):
        freed = C.c_int64()
        _check(lib().swa_radix_evict(self.h, 1 if swa_only else 0, n_tokens, C.byref(freed)), None)
        return freed.value

    def releases(self):
        """(full slots, how many of them still map SWA slots, SWA-only slots)."""
        import numpy as np
        pf, ps_ = C.POINTER(C.c_int64)(), C.POINTER(C.c_int64)()
        nf, nl, ns = C.c_int64(), C.c_int64(), C.c_int64()
        _check(lib().swa_radix_releases(self.h, C.byref(pf), C.byref(nf), C.byref(nl),
                                        C.byref(ps_), C.byref(ns)), None)
        f = np.ctypeslib.as_array(pf, (nf.value,)).copy() if nf.value else np.zeros(0, np.int64)
        s = np.ctypeslib.as_array(ps_, (ns.value,)).copy() if ns.value else np.zeros(0, np.int64)
        return f, nl.value, s

    def sizes(self):
        a, b, c = C.c_int64(), C.c_int64(), C.c_int64()
        _check(lib().swa_radix_sizes(self.h, C.byref(a), C.byref(b), C.byref(c)), None)
        return a.value, b.value, c.value

    def apply_releases(self, ctx, stream=None):
        """Issue the pending releases on ``ctx``: swa_free for full slots,
        swa_free_swa for SWA-only ones, with exact page counts."""
        f, live, s = self.releases()
        ps = self.ps
        if len(f):
            swa_free(ctx, torch.tensor(f, device="cuda"), len(f) // ps, live // ps, stream)
        if len(s):
            swa_free_swa(ctx, torch.tensor(s, device="cuda"), len(s) // ps, stream)
        return f, live, s


def swa_available_size(ctx):
    return lib().swa_available_size(ctx.handle)


def swa_available_full(ctx):
    return lib().swa_available_full(ctx.handle)


def swa_available_swa(ctx):
    return lib().swa_available_swa(ctx.handle)


def swa_device_check(ctx, stream=None):
    err = C.c_int32()
    st = lib().swa_device_check(ctx.handle, _stream(stream), C.byref(err))
    if st not in (SWA_OK, SWA_ERR_DEVICE_CHECK):
        _check(st, ctx.handle)
    return err.value


def swa_sync_counts(ctx, stream=None):
    _check(lib().swa_sync_counts(ctx.handle, _stream(stream)), ctx.handle)


def swa_alloc(ctx, need_size, out_full, out_swa=None, stream=None):
    _check(lib().swa_alloc(ctx.handle, need_size, _ptr(out_full), _ptr(out_swa), _stream(stream)),
           ctx.handle)


def swa_alloc_extend(ctx, prefix_lens, seq_lens, last_loc, prefix_lens_host, seq_lens_host,
                     out_full, out_swa=None, req_to_token=None, req_idx=None, stream=None):
    bs = len(seq_lens_host)
    ph, pp = _host(prefix_lens_host)
    sh, sp = _host(seq_lens_host)
    stride = req_to_token.shape[1] if req_to_token is not None else 0
    _check(lib().swa_alloc_extend(ctx.handle, bs, _ptr(prefix_lens), _ptr(seq_lens), _ptr(last_loc),
                                  pp, sp, _ptr(out_full), _ptr(out_swa), _ptr(req_to_token),
                                  stride, _ptr(req_idx), _stream(stream)), ctx.handle)


def swa_alloc_decode(ctx, seq_lens, last_loc, seq_lens_host, out_full, out_swa=None,
                     req_to_token=None, req_idx=None, stream=None):
    bs = len(seq_lens_host)
    sh, sp = _host(seq_lens_host)
    stride = req_to_token.shape[1] if req_to_token is not None else 0
    _check(lib().swa_alloc_decode(ctx.handle, bs, _ptr(seq_lens), _ptr(last_loc), sp,
                                  _ptr(out_full), _ptr(out_swa), _ptr(req_to_token), stride,
                                  _ptr(req_idx), _stream(stream)), ctx.handle)


def swa_translate(ctx, full_loc, swa_loc, stream=None):
    _check(lib().swa_translate(ctx.handle, _ptr(full_loc), full_loc.numel(), _ptr(swa_loc),
                               _stream(stream)), ctx.handle)


def swa_free(ctx, full_idx, n_full_pages=-1, n_swa_pages=-1, stream=None):
    _check(lib().swa_free(ctx.handle, _ptr(full_idx), full_idx.numel(), n_full_pages, n_swa_pages,
                          _stream(stream)), ctx.handle)


def swa_free_swa(ctx, full_idx, n_swa_pages=-1, stream=None):
    _check(lib().swa_free_swa(ctx.handle, _ptr(full_idx), full_idx.numel(), n_swa_pages,
                              _stream(stream)), ctx.handle)


def swa_evict_swa(ctx, req_to_token, req_idx, pre_lens, evicted, pre_lens_host, evicted_host,
                  protected_lens=None, protected_host=None, interval=0, radix=False, stream=None):
    """``evicted_host`` (numpy int64) is updated in place."""
    bs = len(pre_lens_host)
    ph, pp = _host(pre_lens_host)
    assert isinstance(evicted_host, np.ndarray) and evicted_host.dtype == np.int64
    assert evicted_host.flags["C_CONTIGUOUS"]
    eh = evicted_host.ctypes.data_as(C.c_void_p)
    qh, qp = _host(protected_host)
    _check(lib().swa_evict_swa(ctx.handle, bs, _ptr(req_to_token), req_to_token.shape[1],
                               _ptr(req_idx), _ptr(pre_lens), _ptr(evicted), _ptr(protected_lens),
                               pp, eh, qp, interval, 1 if radix else 0, _stream(stream)),
           ctx.handle)


def swa_store_kv(ctx, layer, k, v, full_loc, swa_loc=None, k_scale=1.0, v_scale=1.0, stream=None):
    _check(lib().swa_store_kv(ctx.handle, layer, _ptr(k), _ptr(v), k.shape[0], _ptr(full_loc),
                              _ptr(swa_loc), k_scale, v_scale, _stream(stream)), ctx.handle)


def swa_plan_bytes(ctx, bs, max_new=1):
    return lib().swa_plan_bytes(ctx.handle, bs, max_new)


def swa_plan(ctx, req_to_token, req_idx, prefix_lens, seq_lens, plan, max_new=1, stream=None):
    bs = seq_lens.numel()
    _check(lib().swa_plan(ctx.handle, bs, _ptr(req_to_token), req_to_token.shape[1], _ptr(req_idx),
                          _ptr(prefix_lens), _ptr(seq_lens), max_new, _ptr(plan), plan.numel(),
                          _stream(stream)), ctx.handle)


def swa_attn_decode_ws_bytes(ctx, layer, bs, max_seq_len):
    return lib().swa_attn_decode_ws_bytes(ctx.handle, layer, bs, max_seq_len)


def swa_attn_decode(ctx, layer, req_to_token, req_idx, seq_lens, max_seq_len, plan, q, sinks,
                    sm_scale, out, ws, k_scale=1.0, v_scale=1.0, stream=None):
    bs = seq_lens.numel()
    stride = req_to_token.shape[1] if req_to_token is not None else 0
    _check(lib().swa_attn_decode(ctx.handle, layer, bs, _ptr(req_to_token), stride, _ptr(req_idx),
                                 _ptr(seq_lens), max_seq_len, _ptr(plan), _ptr(q), _ptr(sinks),
                                 sm_scale, k_scale, v_scale, _ptr(out), _ptr(ws), ws.numel(),
                                 _stream(stream)), ctx.handle)


def swa_store_kv_attn_decode(ctx, layer, req_to_token, req_idx, seq_lens, max_seq_len, plan, q,
                             k_new, v_new, full_loc, swa_loc, sinks, sm_scale, out, ws,
                             k_scale=1.0, v_scale=1.0, stream=None):
    """swa_store_kv of the new tokens, then swa_attn_decode (one launch on the
    tensor-core decode path)."""
    bs = seq_lens.numel()
    stride = req_to_token.shape[1] if req_to_token is not None else 0
    _check(lib().swa_store_kv_attn_decode(ctx.handle, layer, bs, _ptr(req_to_token), stride,
                                          _ptr(req_idx), _ptr(seq_lens), max_seq_len, _ptr(plan),
                                          _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(full_loc),
                                          _ptr(swa_loc), _ptr(sinks), sm_scale, k_scale, v_scale,
                                          _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           ctx.handle)


def swa_attn_decode_noalloc_max_bytes():
    return lib().swa_attn_decode_noalloc_max_bytes()


def swa_attn_decode_noalloc(ctx, layer, req_to_token, req_idx, seq_lens, max_seq_len, plan, q,
                            sinks, sm_scale, out, k_scale=1.0, v_scale=1.0, stream=None):
    """Decode attention with the library's fixed internal scratch (no workspace)."""
    bs = seq_lens.numel()
    stride = req_to_token.shape[1] if req_to_token is not None else 0
    _check(lib().swa_attn_decode_noalloc(ctx.handle, layer, bs, _ptr(req_to_token), stride,
                                         _ptr(req_idx), _ptr(seq_lens), max_seq_len, _ptr(plan),
                                         _ptr(q), _ptr(sinks), sm_scale, k_scale, v_scale,
                                         _ptr(out), _stream(stream)), ctx.handle)


def swa_attn_extend_ws_bytes(ctx, layer, n_tokens, max_seq_len):
    return lib().swa_attn_extend_ws_bytes(ctx.handle, layer, n_tokens, max_seq_len)


def swa_attn_extend(ctx, layer, req_to_token, req_idx, prefix_lens, seq_lens, qo_indptr,
                    n_tokens, max_new, max_seq_len, plan, q, sinks, sm_scale, out, ws,
                    k_scale=1.0, v_scale=1.0, stream=None):
    bs = seq_lens.numel()
    stride = req_to_token.shape[1] if req_to_token is not None else 0
    _check(lib().swa_attn_extend(ctx.handle, layer, bs, _ptr(req_to_token), stride, _ptr(req_idx),
                                 _ptr(prefix_lens), _ptr(seq_lens), _ptr(qo_indptr), n_tokens,
                                 max_new, max_seq_len, _ptr(plan), _ptr(q), _ptr(sinks), sm_scale,
                                 k_scale, v_scale, _ptr(out), _ptr(ws), ws.numel(),
                                 _stream(stream)), ctx.handle)


def swa_last_attn_path(ctx):
    return lib().swa_last_attn_path(ctx.handle)


def swa_set_attn_path(ctx, path):
    _check(lib().swa_set_attn_path(ctx.handle, path), ctx.handle)


def swa_synth_tokens(seed, stream_id, layer, req, pos, heads, dim, out, stream=None):
    dt = DTYPE_F32 if out.dtype == torch.float32 else DTYPE_BF16
    _check(lib().swa_synth_tokens(seed, stream_id, layer, _ptr(req), _ptr(pos), req.numel(), heads,
                                  dim, dt, _ptr(out), _stream(stream)), None)


# ------------------------------------------------- unified pool (two ends) ---
UCTR_LOW, UCTR_HIGH, UCTR_REL_FULL, UCTR_REL_SWA, UCTR_VHEAD, UCTR_VCOUNT, UCTR_ERROR = range(7)


class swa_unified_view(C.Structure):
    _fields_ = [("v2p_full", C.c_void_p), ("v2p_swa", C.c_void_p),
                ("released_full", C.c_void_p), ("released_swa", C.c_void_p),
                ("virt_free", C.c_void_p), ("counters", C.c_void_p), ("num_pages", C.c_int64)]


def _ucheck(status, handle):
    if status != SWA_OK:
        msg = lib().swa_unified_last_error(handle)
        msg = msg.decode() if msg else ""
        cls = SwaNoMem if status == SWA_ERR_NOMEM else SwaError
        raise cls(status, msg)


class UnifiedPool:
    """Owns a swa_unified allocator and its device state blob."""

    def __init__(self, num_pages, page_size, max_batch=64, device="cuda", stream=None):
        n = lib().swa_unified_state_bytes(num_pages, max_batch)
        if n == 0:
            raise SwaError(SWA_ERR_INVALID, "bad unified pool size")
        self.state = torch.empty(n, dtype=torch.uint8, device=device)
        self.num_pages, self.page_size = int(num_pages), int(page_size)
        h = C.c_void_p()
        _ucheck(lib().swa_unified_create(num_pages, page_size, max_batch, _ptr(self.state),
                                         _stream(stream), C.byref(h)), None)
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None):
            lib().swa_unified_destroy(self.handle)
            self.handle = None

    def _view(self):
        v = swa_unified_view()
        _ucheck(lib().swa_unified_state_pointers(self.handle, C.byref(v)), self.handle)
        return v

    def _tensor(self, ptr, n, dtype):
        base = self.state.data_ptr()
        off = ptr - base
        item = torch.tensor([], dtype=dtype).element_size()
        return self.state[off:off + n * item].view(dtype)

    def v2p(self, full: bool):
        v = self._view()
        return self._tensor(v.v2p_full if full else v.v2p_swa, self.num_pages + 1, torch.int64)

    def released(self, full: bool):
        """Released page ids of one side, ascending (from its bitmap)."""
        v = self._view()
        words = (self.num_pages + 1 + 31) // 32
        bm = self._tensor(v.released_full if full else v.released_swa, words, torch.int32)
        bits = bm.cpu().numpy().view(np.uint32)
        return [w * 32 + b for w in range(words) for b in range(32) if (int(bits[w]) >> b) & 1]

    def counters(self):
        v = self._view()
        return self._tensor(v.counters, 8, torch.int64).cpu().tolist()

    def virt_free(self):
        """Free virtual page ids, front first."""
        c = self.counters()
        v = self._view()
        ring = self._tensor(v.virt_free, self.num_pages, torch.int64).cpu().tolist()
        head, count = c[UCTR_VHEAD], c[UCTR_VCOUNT]
        return [ring[(head + i) % self.num_pages] for i in range(count)]


def swa_unified_available_size(u):
    return lib().swa_unified_available_size(u.handle)


def swa_unified_sync(u, stream=None):
    _ucheck(lib().swa_unified_sync(u.handle, _stream(stream)), u.handle)


def swa_unified_device_check(u, stream=None):
    err = C.c_int32()
    st = lib().swa_unified_device_check(u.handle, _stream(stream), C.byref(err))
    if st not in (SWA_OK, SWA_ERR_DEVICE_CHECK):
        _ucheck(st, u.handle)
    return err.value


def swa_unified_alloc_extend(u, prefix_lens, seq_lens, last_loc, prefix_lens_host, seq_lens_host,
                             out_virt, req_to_token=None, req_idx=None, stream=None):
    bs = len(seq_lens_host)
    ph, pp = _host(prefix_lens_host)
    sh, sp = _host(seq_lens_host)
    rt_stride = req_to_token.shape[1] if req_to_token is not None else 0
    _ucheck(lib().swa_unified_alloc_extend(u.handle, bs, _ptr(prefix_lens), _ptr(seq_lens),
                                           _ptr(last_loc), pp, sp, _ptr(out_virt),
                                           _ptr(req_to_token), rt_stride, _ptr(req_idx),
                                           _stream(stream)), u.handle)


def swa_unified_free_swa(u, virt, stream=None):
    _ucheck(lib().swa_unified_free_swa(u.handle, _ptr(virt), virt.numel(), _stream(stream)),
            u.handle)


def swa_unified_free(u, virt, stream=None):
    _ucheck(lib().swa_unified_free(u.handle, _ptr(virt), virt.numel(), _stream(stream)), u.handle)


def swa_unified_evict_swa(u, window_excl, req_to_token, req_idx, pre_lens, evicted, pre_lens_host,
                          evicted_host, protected_lens=None, protected_host=None, interval=0,
                          radix=False, stream=None):
    """``evicted_host`` (numpy int64) is updated in place."""
    bs = len(pre_lens_host)
    ph, pp = _host(pre_lens_host)
    assert isinstance(evicted_host, np.ndarray) and evicted_host.dtype == np.int64
    assert evicted_host.flags["C_CONTIGUOUS"]
    prh, prp = _host(protected_host)
    _ucheck(lib().swa_unified_evict_swa(u.handle, bs, window_excl, _ptr(req_to_token),
                                        req_to_token.shape[1], _ptr(req_idx), _ptr(pre_lens),
                                        _ptr(evicted), _ptr(protected_lens), pp,
                                        evicted_host.ctypes.data_as(C.c_void_p), prp, interval,
                                        1 if radix else 0, _stream(stream)), u.handle)
