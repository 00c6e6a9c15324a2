"""Drives the CUDA path (through the C-ABI binding) and the oracle side by side
on the same seeded inputs, and compares what they produce.

Used only by tests.  GPU and oracle share nothing but the inputs drawn from
``hybrid_sliding_window_gb300.synth``.
"""
from __future__ import annotations

import numpy as np
import torch

from hybrid_sliding_window_gb300 import api, synth
from oracle import allocator as OA
from oracle import attention as OT
from oracle import kvstore as OK

DT = {"f32": api.DTYPE_F32, "bf16": api.DTYPE_BF16, "e4m3": api.DTYPE_E4M3}
KIND = {OT.FULL: api.LAYER_FULL, OT.SLIDING: api.LAYER_SLIDING, OT.CHUNKED: api.LAYER_CHUNKED}
ITEM = {"f32": 4, "bf16": 2, "e4m3": 1}
TOL = {"f32": 1e-5, "bf16": 2e-2, "e4m3": 2e-2}


def envelope_bytes(size, ps, n_layers, row_bytes):
    pages = size // ps + 1
    return (pages * 2 * n_layers * ps + 2 * n_layers * ps) * row_bytes


class Pair:
    """One model configuration instantiated on the GPU and in the oracle."""

    def __init__(self, layers, Hq, D, dtype, ps, size_full, size_swa, layout="per_layer",
                 need_sort=False, seed=0, perm_free=False, max_batch=64, max_ctx=512,
                 max_reqs=8, k_scale=1.0, v_scale=1.0, oracle=True, ring_size=0):
        self.layers = layers          # list of (kind, window, hkv)
        self.ring = ring_size > 0     # per-request SWA rings, one per req_to_token row
        if self.ring:
            size_swa = OA.ring_pool_size(max_reqs + 1, ring_size, ps)
        self.Hq, self.D, self.dtype, self.ps = Hq, D, dtype, ps
        self.seed = seed
        self.k_scale, self.v_scale = k_scale, v_scale
        self.lookback = max([OT.lookback(k, w) for k, w, _ in layers if k != OT.FULL] or [0])
        dev = "cuda"
        init_f = init_s = None
        if perm_free:
            init_f = synth.permutation(seed + 101, size_full // ps)
            init_s = synth.permutation(seed + 202, size_swa // ps)
        store_t = api._STORE_TORCH[DT[dtype]]
        self.kv = []
        gl = []
        full_env = swa_env = None
        if layout == "per_layer":
            for kind, w, hkv in layers:
                n = (size_full if kind == OT.FULL else size_swa) + ps
                k = torch.zeros((n, hkv, D), dtype=store_t, device=dev)
                v = torch.zeros((n, hkv, D), dtype=store_t, device=dev)
                self.kv.append((k, v))
                gl.append(dict(kind=KIND[kind], window=w, num_kv_heads=hkv, k=k, v=v))
        else:
            nf = sum(1 for k, _, _ in layers if k == OT.FULL)
            nsw = len(layers) - nf
            hf = [h for k, _, h in layers if k == OT.FULL]
            hs = [h for k, _, h in layers if k != OT.FULL]
            if nf:
                full_env = torch.zeros(envelope_bytes(size_full, ps, nf, hf[0] * D * ITEM[dtype]),
                                       dtype=torch.uint8, device=dev)
            if nsw:
                swa_env = torch.zeros(envelope_bytes(size_swa, ps, nsw, hs[0] * D * ITEM[dtype]),
                                      dtype=torch.uint8, device=dev)
            for kind, w, hkv in layers:
                gl.append(dict(kind=KIND[kind], window=w, num_kv_heads=hkv))
        self.ctx = api.SwaCtx(gl, ps, size_full, size_swa, Hq, D, DT[dtype],
                              api.LAYOUT_PER_LAYER if layout == "per_layer" else api.LAYOUT_ENVELOPE,
                              need_sort, max_batch, full_env, swa_env,
                              torch.tensor(init_f, device=dev) if init_f is not None else None,
                              torch.tensor(init_s, device=dev) if init_s is not None else None,
                              ring_size=ring_size, ring_slots=(max_reqs + 1) if self.ring else 0)
        self.rt = torch.zeros((max_reqs + 1, max_ctx), dtype=torch.int32, device=dev)
        self.oracle = oracle
        if oracle:
            if self.ring:
                self.oa = OA.RingTwoPoolAllocator(size_full, ps, ring_size, max_reqs + 1,
                                                  self.lookback, need_sort, init_f)
            else:
                self.oa = OA.TwoPoolAllocator(size_full, size_swa, ps, need_sort, init_f, init_s)
            self.op = OK.OraclePools(layers, size_full, size_swa, ps, D, dtype, layout)
            self.ort = np.zeros((max_reqs + 1, max_ctx), dtype=np.int64)
        self.sinks = [synth.sinks(seed, l, Hq) for l in range(len(layers))]
        self.sinks_d = [torch.tensor(s, device=dev) for s in self.sinks]
        self.scale = 1.0 / np.sqrt(D)
        # Optional input shaping for wide score ranges: q is multiplied by
        # q_gain, the K rows of position t by k_gain(t); the products are
        # rounded to the input dtype, so both sides read the same values.
        self.q_gain = 1.0
        self.k_gain = None

    def set_sinks(self, l, values):
        self.sinks[l] = np.asarray(values, np.float32)
        self.sinks_d[l] = torch.tensor(self.sinks[l], device="cuda")

    # ------------------------------------------------------------- inputs ---
    def kv_in(self, l, reqs, pos):
        hkv = self.layers[l][2]
        bf = self.dtype != "f32"
        k = synth.tokens(self.seed, synth.STREAM_K, l, reqs, pos, hkv, self.D, bf16=bf)
        v = synth.tokens(self.seed, synth.STREAM_V, l, reqs, pos, hkv, self.D, bf16=bf)
        if self.k_gain is not None:
            g = np.asarray(self.k_gain(np.asarray(pos, np.int64)), np.float32).reshape(-1, 1, 1)
            k = (k * g).astype(np.float32)
            k = synth.to_bf16_values(k) if bf else k
        return k, v

    def q_in(self, l, reqs, pos):
        bf = self.dtype != "f32"
        q = synth.tokens(self.seed, synth.STREAM_Q, l, reqs, pos, self.Hq, self.D, bf16=bf)
        if self.q_gain != 1.0:
            q = (q * np.float32(self.q_gain)).astype(np.float32)
            q = synth.to_bf16_values(q) if bf else q
        return q

    def to_dev(self, x):
        t = torch.tensor(x, device="cuda")
        return t.to(torch.bfloat16) if self.dtype != "f32" else t

    # -------------------------------------------------------------- steps ---
    def extend(self, rows, pre, seq, check_alloc=True, store=True):
        """Allocate + store positions pre..seq-1 of request rows (row ids of
        req_to_token; request id for the generator = row).  store=False
        allocates only (a decode step whose attention call stores the token)."""
        rows = list(rows)
        pre = np.asarray(pre, np.int64)
        seq = np.asarray(seq, np.int64)
        n = int((seq - pre).sum())
        out_f = torch.empty(n, dtype=torch.int64, device="cuda")
        out_s = torch.empty(n, dtype=torch.int64, device="cuda")
        d_pre = torch.tensor(pre, device="cuda")
        d_seq = torch.tensor(seq, device="cuda")
        d_rows = torch.tensor(rows, dtype=torch.int64, device="cuda")
        api.swa_alloc_extend(self.ctx, d_pre, d_seq, None, pre, seq, out_f, out_s,
                             req_to_token=self.rt, req_idx=d_rows)
        reqs = [r for r, p, s in zip(rows, pre, seq) for _ in range(p, s)]
        pos = [t for r, p, s in zip(rows, pre, seq) for t in range(p, s)]
        if self.oracle:
            last = [int(self.ort[r, p - 1]) if p > 0 else -1 for r, p in zip(rows, pre)]
            if self.ring:
                of, osw = self.oa.alloc_extend(pre, seq, last, rows)
            else:
                of, osw = self.oa.alloc_extend(pre, seq, last)
            for i, (r, t) in enumerate(zip(reqs, pos)):
                self.ort[r, t] = of[i]
            if check_alloc:
                np.testing.assert_array_equal(out_f.cpu().numpy(), np.array(of, np.int64))
                np.testing.assert_array_equal(out_s.cpu().numpy(), np.array(osw, np.int64))
        if self.oracle:
            self.last_alloc = (of, osw)
        for l in range(len(self.layers) if store else 0):
            k, v = self.kv_in(l, reqs, pos)
            api.swa_store_kv(self.ctx, l, self.to_dev(k), self.to_dev(v), out_f, out_s,
                             self.k_scale, self.v_scale)
            if self.oracle:
                self.op.store(l, k, v, of, osw, self.k_scale, self.v_scale)
        return out_f, out_s

    def evict(self, rows, pre, evicted_h, interval, protected=None):
        rows = list(rows)
        pre = np.asarray(pre, np.int64)
        ev_before = evicted_h.copy()
        d_ev = torch.tensor(evicted_h, device="cuda")
        prot_d = torch.tensor(protected, device="cuda") if protected is not None else None
        api.swa_evict_swa(self.ctx, self.rt, torch.tensor(rows, dtype=torch.int64, device="cuda"),
                          torch.tensor(pre, device="cuda"), d_ev, pre, evicted_h,
                          protected_lens=prot_d, protected_host=protected, interval=interval)
        np.testing.assert_array_equal(d_ev.cpu().numpy(), evicted_h)
        if self.oracle:
            o_ev, _ = OA.evict_swa(self.oa, self.ort, rows, pre, ev_before,
                                   protected if protected is not None else [0] * len(rows),
                                   self.lookback, interval)
            np.testing.assert_array_equal(np.array(o_ev, np.int64), evicted_h)
        return evicted_h

    def decode_attention(self, rows, seq, layers=None, max_seq_len=None, new_slots=None):
        """Query at seq-1 (KV stored).  Returns {layer: (gpu, oracle)}.
        new_slots=(out_f, out_s) from extend(..., store=False): the token at
        seq-1 is not stored yet; each layer's swa_store_kv_attn_decode stores
        it (the oracle stores it first)."""
        rows = list(rows)
        seq = np.asarray(seq, np.int64)
        bs = len(rows)
        d_seq = torch.tensor(seq, device="cuda")
        d_rows = torch.tensor(rows, dtype=torch.int64, device="cuda")
        plan = torch.zeros(api.swa_plan_bytes(self.ctx, bs, 1), dtype=torch.uint8, device="cuda")
        api.swa_plan(self.ctx, self.rt, d_rows, None, d_seq, plan, 1)
        msl = int(max_seq_len or seq.max())
        res = {}
        for l in (layers if layers is not None else range(len(self.layers))):
            q = self.q_in(l, rows, seq - 1)
            qd = self.to_dev(q)
            out = torch.empty_like(qd)
            ws = torch.zeros(api.swa_attn_decode_ws_bytes(self.ctx, l, bs, msl), dtype=torch.uint8,
                             device="cuda")
            if new_slots is None:
                api.swa_attn_decode(self.ctx, l, self.rt, d_rows, d_seq, msl, plan, qd,
                                    self.sinks_d[l], self.scale, out, ws, self.k_scale,
                                    self.v_scale)
            else:
                k, v = self.kv_in(l, rows, list(seq - 1))
                if self.oracle:
                    of, osw = self.last_alloc
                    self.op.store(l, k, v, of, osw, self.k_scale, self.v_scale)
                api.swa_store_kv_attn_decode(self.ctx, l, self.rt, d_rows, d_seq, msl, plan, qd,
                                             self.to_dev(k), self.to_dev(v), new_slots[0],
                                             new_slots[1], self.sinks_d[l], self.scale, out, ws,
                                             self.k_scale, self.v_scale)
            g = out.float().cpu().numpy()
            o = None
            if self.oracle:
                o = OK.attention_through_tables(
                    self.op, self.oa, l, self.ort, rows,
                    [(b, int(s) - 1) for b, s in enumerate(seq)],
                    q, self.sinks[l], self.scale, self.k_scale, self.v_scale)
            res[l] = (g, o)
        return res

    def extend_attention(self, rows, pre, seq, layers=None):
        rows = list(rows)
        pre = np.asarray(pre, np.int64)
        seq = np.asarray(seq, np.int64)
        bs = len(rows)
        ext = seq - pre
        indptr = np.concatenate([[0], np.cumsum(ext)]).astype(np.int64)
        n = int(indptr[-1])
        d = lambda x: torch.tensor(x, device="cuda")
        d_rows = torch.tensor(rows, dtype=torch.int64, device="cuda")
        max_new = int(ext.max())
        plan = torch.zeros(api.swa_plan_bytes(self.ctx, bs, max_new), dtype=torch.uint8, device="cuda")
        api.swa_plan(self.ctx, self.rt, d_rows, d(pre), d(seq), plan, max_new)
        reqs = [r for r, p, s in zip(rows, pre, seq) for _ in range(p, s)]
        pos = [t for r, p, s in zip(rows, pre, seq) for t in range(p, s)]
        res = {}
        for l in (layers if layers is not None else range(len(self.layers))):
            q = self.q_in(l, reqs, pos)
            qd = self.to_dev(q)
            out = torch.empty_like(qd)
            msl = int(seq.max())
            ws = torch.zeros(api.swa_attn_extend_ws_bytes(self.ctx, l, n, msl), dtype=torch.uint8,
                             device="cuda")
            api.swa_attn_extend(self.ctx, l, self.rt, d_rows, d(pre), d(seq), d(indptr), n, max_new,
                                msl, plan, qd, self.sinks_d[l], self.scale, out, ws,
                                self.k_scale, self.v_scale)
            g = out.float().cpu().numpy()
            o = None
            if self.oracle:
                bidx = [b for b in range(bs) for _ in range(int(ext[b]))]
                o = OK.attention_through_tables(
                    self.op, self.oa, l, self.ort, rows, list(zip(bidx, pos)), q,
                    self.sinks[l], self.scale, self.k_scale, self.v_scale)
            res[l] = (g, o)
        return res

    # --------------------------------------------------------- comparison ---
    def check_state(self):
        """Mapping, free lists, req_to_token and stored KV bytes: bit exact."""
        assert self.oracle
        torch.cuda.synchronize()
        assert api.swa_device_check(self.ctx) == 0
        np.testing.assert_array_equal(self.ctx.mapping().cpu().numpy(),
                                      np.array(self.oa.mapping, np.int64))
        for full, led in ((True, self.oa.full), (False, self.oa.swa)):
            if not full and self.ring:
                continue          # rings: the SWA free list is never touched
            free, staged = self.ctx.free_list(full)
            assert free == led.free
            assert sorted(staged) == sorted(p for s in led.staged for p in s)
        np.testing.assert_array_equal(self.rt.cpu().numpy().astype(np.int64), self.ort)
        assert api.swa_available_full(self.ctx) == self.oa.full.available_size()
        assert api.swa_available_swa(self.ctx) == self.oa.swa.available_size()
        assert api.swa_available_size(self.ctx) == self.oa.available_size()
        self.check_kv_bytes()

    def check_kv_bytes(self):
        if self.op.layout == "per_layer":
            for l, (k, v) in enumerate(self.kv):
                for dev_t, host in ((k, self.op.k[l]), (v, self.op.v[l])):
                    d = dev_t.cpu()
                    if d.dtype == torch.bfloat16:
                        d = d.view(torch.int16).numpy().view(np.uint16)
                    else:
                        d = d.numpy()
                    np.testing.assert_array_equal(d, host)
        else:
            for is_full, buf in ((True, self.ctx.full_envelope), (False, self.ctx.swa_envelope)):
                if buf is None:
                    continue
                np.testing.assert_array_equal(buf.cpu().numpy(), self.op.raw[is_full])


def assert_close(gpu, ref, tol, what=""):
    ref = np.asarray(ref, np.float64)
    gpu = np.asarray(gpu, np.float64)
    bad = np.abs(gpu - ref) > tol + tol * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tol {tol}; first at "
                             f"{tuple(i)}: gpu={gpu[tuple(i)]} ref={ref[tuple(i)]}")


# ---------------------------------------------------------------------------
# Trace replay for workloads built by hybrid_sliding_window_gb300.workloads
# ---------------------------------------------------------------------------
from hybrid_sliding_window_gb300.workloads import CHUNKED, FULL, SLIDING  # noqa: E402
from oracle import codecs as OC  # noqa: E402

OKIND = {FULL: OT.FULL, SLIDING: OT.SLIDING, CHUNKED: OT.CHUNKED}


def replay(st: DecodeState):
    """The oracle allocator driven by the GPU state's recorded calls."""
    spec = st.spec
    init_f = init_s = None
    if spec.perm_free:      # the same seeded page order the GPU state was given
        init_f = synth.permutation(spec.seed + 101, st.size_full // spec.ps)
        init_s = synth.permutation(spec.seed + 202, st.size_swa // spec.ps)
    if st.swa_ring:
        oa = OA.RingTwoPoolAllocator(st.size_full, spec.ps, st.ring_size, st.B + 1, spec.lookback(),
                                     False, init_f)
    else:
        oa = OA.TwoPoolAllocator(st.size_full, st.size_swa, spec.ps, False, init_f, init_s)
    ort = np.zeros(tuple(st.rt.shape), np.int64)
    for op in st.trace:
        if op[0] == "evict":
            _, rows, pre, ev, interval = op
            OA.evict_swa(oa, ort, rows, pre, ev, [0] * len(rows), spec.lookback(), interval)
        else:
            if op[0] == "extend":
                _, rows, pre, seq = op
            else:
                _, rows, seq = op
                pre = [s - 1 for s in seq]
            last = [int(ort[r, p - 1]) if p > 0 else -1 for r, p in zip(rows, pre)]
            if st.swa_ring:
                full, _ = oa.alloc_extend(pre, seq, last, rows)
            else:
                full, _ = oa.alloc_extend(pre, seq, last)
            off = 0
            for r, p, s in zip(rows, pre, seq):
                ort[r, p:s] = full[off:off + s - p]
                off += s - p
    return oa, ort


def check_state(st, oa, ort):
    torch.cuda.synchronize()
    assert api.swa_device_check(st.ctx) == 0
    np.testing.assert_array_equal(st.ctx.mapping().cpu().numpy(), np.array(oa.mapping, np.int64))
    for full, led in ((True, oa.full), (False, oa.swa)):
        if not full and st.swa_ring:
            continue          # rings: the SWA free list is never touched
        free, _ = st.ctx.free_list(full)
        assert free == led.free
    np.testing.assert_array_equal(st.rt.cpu().numpy().astype(np.int64), ort)
    assert api.swa_available_size(st.ctx) == oa.available_size()


def oracle_decode(st, oa, ort, layer, b, seq_b, q_row):
    """Oracle output [Hq, D] for batch entry b at position seq_b - 1."""
    spec = st.spec
    kind, w, hkv = spec.layers[layer]
    p = int(seq_b) - 1
    row = int(st.rows[b])
    J = list(OT.key_positions(OKIND[kind], w, p))
    if kind != FULL:
        assert all(oa.mapping[int(ort[row, j])] > 0 for j in J), "evicted key in window"
    bf = spec.dtype != "f32"
    K = synth.tokens(spec.seed, synth.STREAM_K, layer, [row] * len(J), J, hkv, spec.D, bf16=bf)
    V = synth.tokens(spec.seed, synth.STREAM_V, layer, [row] * len(J), J, hkv, spec.D, bf16=bf)
    if spec.dtype == "e4m3":
        K = OC.e4m3_decode(OC.e4m3_encode(K))
        V = OC.e4m3_decode(OC.e4m3_encode(V))
    return OT.attend_heads(q_row.astype(np.float64), K, V, st.sinks_h[layer], st.scale)


