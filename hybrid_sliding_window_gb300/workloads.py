"""Seeded synthetic workloads shaped like the pages' hybrid models, and a GPU
decode state that builds its KV cache by replaying the method itself.

Model shapes ("SWA in SGLang" design note, "design"): MiMo-V2-Flash (48
layers, 39 sliding with window 128 and 8 KV heads, 9 full with 4 KV heads),
GPT-OSS (sliding and full layers alternating), Llama4 (3 of every 4 layers
chunked-local, the 4th global).  The pages do not give MiMo's
hybrid_layer_pattern; full layers sit at every 5th position from layer 4.

Everything here calls the C library through ``api``; inputs (q, k, v,
sinks) come from ``synth``.  The state keeps a trace of the allocation /
eviction calls it made so that a test can replay the same sequence on the
CPU oracle.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from . import api, synth

FULL, SLIDING, CHUNKED = api.LAYER_FULL, api.LAYER_SLIDING, api.LAYER_CHUNKED
DTYPES = {"f32": api.DTYPE_F32, "bf16": api.DTYPE_BF16, "e4m3": api.DTYPE_E4M3}
ESIZE = {"f32": 4, "bf16": 2, "e4m3": 1}


def mimo_layers():
    return [(FULL, 0, 4) if l % 5 == 4 else (SLIDING, 127, 8) for l in range(48)]


def gptoss_layers():
    return [(SLIDING, 127, 8) if l % 2 == 0 else (FULL, 0, 8) for l in range(24)]


def llama4_layers(groups=12):
    return [(FULL, 0, 8) if l % 4 == 3 else (CHUNKED, 8192, 8) for l in range(4 * groups)]


@dataclasses.dataclass
class Spec:
    name: str
    layers: list
    Hq: int
    D: int
    dtype: str
    ps: int
    batch: int
    seq_kind: str            # "uniform", "loguniform", "fixed"
    seq_lo: int
    seq_hi: int
    r: float
    interval: int
    seed: int
    layout: str = "per_layer"
    sinks: bool = True
    chunk: int = 8192
    description: str = ""
    seq_list: tuple = None   # explicit lengths (overrides seq_kind)
    pools: tuple = None      # (size_full, size_swa) in tokens instead of the sizing rule
    perm_free: bool = False  # pages handed out in a seeded permuted order

    def seq_lens(self) -> np.ndarray:
        if self.seq_list is not None:
            return np.asarray(self.seq_list, dtype=np.int64)
        if self.seq_kind == "uniform":
            return synth.seq_lens_uniform(self.seed, self.batch, self.seq_lo, self.seq_hi)
        if self.seq_kind == "loguniform":
            return synth.seq_lens_log_uniform(self.seed, self.batch, self.seq_lo, self.seq_hi)
        return np.full(self.batch, self.seq_lo, dtype=np.int64)

    def lookback(self) -> int:
        lb = 0
        for kind, w, _ in self.layers:
            if kind == SLIDING:
                lb = max(lb, w)
            elif kind == CHUNKED:
                lb = max(lb, w - 1)
        return lb


EXTEND_SPEC = Spec("extend", mimo_layers(), 64, 128, "bf16", 64, 4, "fixed", 24577, 24577, 0.8,
                   128, 3, description="Chunked-prefill extend, MiMo-shaped layers: B=4 requests, "
                   "24576-token cached prefix + one 8192-token chunk each, W=128, bf16 KV, page 64; "
                   "SWA KV evicted below the window before the chunk")
EXTEND_PREFIX = 24576
EXTEND_CHUNK = 8192

SPECS = {
    "tiny": Spec("tiny", [(SLIDING, 15, 1), (FULL, 0, 1)], 4, 64, "f32", 1, 2, "fixed", 0, 0, 0.25,
                 8, 0, chunk=32, seq_list=(37, 200), pools=(512, 128), perm_free=True,
                 description="Tiny: 1 sliding (W=16) + 1 full layer, 4 query heads, 1 KV head, D=64, "
                 "fp32 KV, page 1, full pool 512 / SWA pool 128 slots in seeded permuted order, "
                 "2 decode requests at seqlens 37 and 200, eviction interval 8"),
    "mimo": Spec("mimo", mimo_layers(), 64, 128, "bf16", 64, 64, "uniform", 4096, 32768, 0.8,
                 128, 1, description="MiMo-V2-Flash-shaped decode: 48 layers (39 sliding W=128 "
                 "with 8 KV heads, 9 full with 4 KV heads), 64 query heads, D=128, bf16 KV, "
                 "page 64, B=64, seqlens U[4096,32768], r=0.8, eviction interval 128"),
    "gptoss": Spec("gptoss", gptoss_layers(), 64, 64, "bf16", 16, 128, "loguniform", 1024, 16384,
                   0.8, 128, 2, description="GPT-OSS-shaped decode: 24 layers alternating "
                   "sliding (W=128) and full, 64 query heads, 8 KV heads, D=64, bf16 KV, page 16, "
                   "B=128, seqlens log-uniform [1024,16384], r=0.8"),
    "llama4": Spec("llama4", llama4_layers(), 40, 128, "e4m3", 64, 16, "fixed", 131072, 131072,
                   0.05, 128, 4, layout="envelope", sinks=False, description="Llama4-shaped "
                   "long-context decode: 12 x [3 chunked-local (C=8192) + 1 global] layers, 40 "
                   "query heads, 8 KV heads, D=128, FP8-E4M3 KV in the page-major envelope, page 64, "
                   "B=16 at seqlen 131072, r=0.05"),
}


def sizing(spec: Spec, seq: np.ndarray, headroom: int):
    """Pool sizes by the pages' rule: cell = F*L_full + r*S*L_swa, with the
    memory budget chosen as cell * N_full for the full-pool need, raised if
    the SWA pool would not hold the prefill's live window."""
    ps = spec.ps
    es = ESIZE[spec.dtype]
    full_h = [h for k, _, h in spec.layers if k == FULL]
    swa_h = [h for k, _, h in spec.layers if k != FULL]
    F = (full_h[0] if full_h else 0) * 2 * spec.D * es
    S = (swa_h[0] if swa_h else 0) * 2 * spec.D * es
    Lf, Ls = len(full_h), len(swa_h)
    n_full = int(sum(math.ceil((int(s) + headroom) / ps) * ps + ps for s in seq))
    lb = spec.lookback()
    # Live SWA slots at the prefill peak (one request group at a time).
    swa_min = spec.batch * (lb + spec.interval + 3 * ps) + spec.chunk + lb + 2 * ps
    n_full = max(n_full, int(math.ceil(swa_min / spec.r)))
    cell = F * Lf + spec.r * S * Ls
    M = int(math.ceil(cell * (n_full + ps)))
    nf, ns = api.swa_pool_sizes(M, F, S, Lf, Ls, spec.r, ps, lb)
    return nf, ns, M


class DecodeState:
    """A whole decode workload resident on one GPU."""

    def __init__(self, spec: Spec, max_steps: int = 64, device: str = "cuda", trace: bool = False,
                 poison_page0: bool = False, swa_ring: bool = False):
        """``swa_ring``: per-request SWA rings (one per request slot, holding the
        window plus one prefill chunk) instead of the paged SWA pool."""
        self.spec = spec
        self.dev = device
        self.seq0 = spec.seq_lens()
        self.B = spec.batch
        self.max_steps = max_steps
        self.ps = spec.ps
        if spec.pools is not None:
            nf, ns = spec.pools
            M = 0
        else:
            nf, ns, M = sizing(spec, self.seq0, max_steps + spec.interval)
        self.swa_ring = swa_ring
        self.ring_size = 0
        if swa_ring:
            self.ring_size = spec.chunk + spec.lookback()
            cost = -(-self.ring_size // spec.ps) * spec.ps
            ns = (self.B + 1) * cost          # one ring per req_to_token row
        self.size_full, self.size_swa, self.mem_budget = nf, ns, M
        self.max_ctx = int(self.seq0.max()) + max_steps + 2 * spec.ps
        self.max_seq_len = int(self.seq0.max()) + max_steps
        self.trace = [] if trace else None
        st = api._STORE_TORCH[DTYPES[spec.dtype]]
        gl = []
        self.kv = []
        self.full_env = self.swa_env = None
        if spec.layout == "per_layer":
            for kind, w, hkv in spec.layers:
                n = (nf if kind == FULL else ns) + spec.ps
                k = torch.zeros((n, hkv, spec.D), dtype=st, device=device)
                v = torch.zeros((n, hkv, spec.D), dtype=st, device=device)
                if poison_page0:
                    k[:spec.ps].fill_(float("nan")) if st != torch.uint8 else k[:spec.ps].fill_(0x7F)
                    v[:spec.ps].fill_(float("nan")) if st != torch.uint8 else v[:spec.ps].fill_(0x7F)
                self.kv.append((k, v))
                gl.append(dict(kind=kind, window=w, num_kv_heads=hkv, k=k, v=v))
        else:
            lf = sum(1 for k, _, _ in spec.layers if k == FULL)
            ls = len(spec.layers) - lf
            hf = [h for k, _, h in spec.layers if k == FULL][0]
            hs = [h for k, _, h in spec.layers if k != FULL][0]
            rb_f = hf * spec.D * ESIZE[spec.dtype]
            rb_s = hs * spec.D * ESIZE[spec.dtype]
            self.full_env = torch.zeros(((nf // spec.ps + 2) * 2 * lf * spec.ps) * rb_f,
                                        dtype=torch.uint8, device=device)
            self.swa_env = torch.zeros(((ns // spec.ps + 2) * 2 * ls * spec.ps) * rb_s,
                                       dtype=torch.uint8, device=device)
            if poison_page0:
                self.full_env[: 2 * lf * spec.ps * rb_f].fill_(0x7F)
                self.swa_env[: 2 * ls * spec.ps * rb_s].fill_(0x7F)
            for kind, w, hkv in spec.layers:
                gl.append(dict(kind=kind, window=w, num_kv_heads=hkv))
        init_f = init_s = None
        if spec.perm_free:
            init_f = torch.tensor(synth.permutation(spec.seed + 101, nf // spec.ps), device=device)
            init_s = torch.tensor(synth.permutation(spec.seed + 202, ns // spec.ps), device=device)
        self.init_free = (init_f, init_s)
        self.ctx = api.SwaCtx(gl, spec.ps, nf, ns, spec.Hq, spec.D, DTYPES[spec.dtype],
                              api.LAYOUT_PER_LAYER if spec.layout == "per_layer"
                              else api.LAYOUT_ENVELOPE, False, max(self.B, 1),
                              self.full_env, self.swa_env, init_f, init_s, device=device,
                              ring_size=self.ring_size, ring_slots=(self.B + 1) if swa_ring else 0)
        self.rt = torch.zeros((self.B + 1, self.max_ctx), dtype=torch.int32, device=device)
        self.rows = np.arange(1, self.B + 1, dtype=np.int64)
        self.rows_d = torch.tensor(self.rows, device=device)
        self.lens = np.zeros(self.B, np.int64)        # tokens with stored KV
        self.evicted = np.zeros(self.B, np.int64)
        self.evicted_d = torch.zeros(self.B, dtype=torch.int64, device=device)
        self.sinks_h = [synth.sinks(spec.seed, l, spec.Hq) if spec.sinks else None
                        for l in range(len(spec.layers))]
        self.sinks_d = [torch.tensor(s, device=device) if s is not None else None for s in self.sinks_h]
        self.scale = 1.0 / math.sqrt(spec.D)
        self.in_dtype = torch.float32 if spec.dtype == "f32" else torch.bfloat16
        self.stream = torch.cuda.current_stream()
        self.last_launches = 0

    # -- helpers ------------------------------------------------------------
    def _synth(self, stream_id, layer, req_d, pos_d, heads):
        out = torch.empty((req_d.numel(), heads, self.spec.D), dtype=self.in_dtype, device=self.dev)
        api.swa_synth_tokens(self.spec.seed, stream_id, layer, req_d, pos_d, heads, self.spec.D, out)
        return out

    def _evict(self, idx, interval, events=None):
        """Eviction pass over batch entries idx (numpy); ``events`` (start,
        end) are recorded around the library call alone."""
        idx_d = torch.tensor(idx, device=self.dev)
        ev_h = self.evicted[idx].copy()
        ev_d = self.evicted_d[idx_d].contiguous()
        pre = self.lens[idx].copy()
        rows_d = self.rows_d[idx_d].contiguous()
        pre_d = torch.tensor(pre, device=self.dev)
        if self.trace is not None:
            self.trace.append(("evict", self.rows[idx].tolist(), pre.tolist(), ev_h.tolist(), interval))
        if events:
            events[0].record()
        api.swa_evict_swa(self.ctx, self.rt, rows_d, pre_d, ev_d, pre, ev_h, interval=interval)
        if events:
            events[1].record()
        self.evicted[idx] = ev_h
        self.evicted_d[idx_d] = ev_d

    def _extend(self, idx, new_lens):
        """alloc_extend + store of positions lens..new_lens-1 for entries idx."""
        pre = self.lens[idx].copy()
        seq = np.asarray(new_lens, np.int64)
        n = int((seq - pre).sum())
        if self.trace is not None:
            self.trace.append(("extend", self.rows[idx].tolist(), pre.tolist(), seq.tolist()))
        out_f = torch.empty(n, dtype=torch.int64, device=self.dev)
        out_s = torch.empty(n, dtype=torch.int64, device=self.dev)
        idx_d = torch.tensor(idx, device=self.dev)
        api.swa_alloc_extend(self.ctx, torch.tensor(pre, device=self.dev),
                             torch.tensor(seq, device=self.dev), None, pre, seq, out_f, out_s,
                             req_to_token=self.rt, req_idx=self.rows_d[idx_d].contiguous())
        reqs = torch.tensor(np.repeat(self.rows[idx], seq - pre), device=self.dev)
        pos = torch.tensor(np.concatenate([np.arange(p, s) for p, s in zip(pre, seq)]),
                           device=self.dev)
        for l, (kind, w, hkv) in enumerate(self.spec.layers):
            k = self._synth(synth.STREAM_K, l, reqs, pos, hkv)
            v = self._synth(synth.STREAM_V, l, reqs, pos, hkv)
            api.swa_store_kv(self.ctx, l, k, v, out_f, out_s)
        self.lens[idx] = seq

    def prefill(self, prompt=None, final_evict=True):
        """Chunked prefill of every request to ``prompt`` (default seq - 1)
        tokens, evicting out-of-window SWA KV before each chunk; requests
        are admitted in groups the SWA pool can hold."""
        spec = self.spec
        prompt = self.seq0 - 1 if prompt is None else np.asarray(prompt, np.int64)
        per_req = spec.chunk + spec.lookback() + 2 * spec.ps
        rest = spec.lookback() + 2 * spec.ps
        g = max(1, min(self.B, (self.size_swa - self.B * rest) // per_req))
        if self.swa_ring:
            g = self.B                         # every request has its own ring
        for g0 in range(0, self.B, g):
            grp = np.arange(g0, min(self.B, g0 + g))
            while (self.lens[grp] < prompt[grp]).any():
                sel = grp[self.lens[grp] < prompt[grp]]
                self._evict(sel, 0)
                self._extend(sel, np.minimum(self.lens[sel] + spec.chunk, prompt[sel]))
            # A finished prompt keeps only its window (what the first decode
            # step's eviction would leave), so the next group fits.
            if final_evict:
                self._evict(grp, 0)
        torch.cuda.synchronize()

    # -- decode -----------------------------------------------------------------
    def make_decode_inputs(self, n_steps: int):
        """q/k/v of n_steps decode steps for every layer, drawn on the device."""
        spec = self.spec
        steps = []
        for s in range(n_steps):
            pos = torch.tensor(self.lens + s, device=self.dev)   # position of the new token
            reqs = self.rows_d
            q, k, v = [], [], []
            for l, (kind, w, hkv) in enumerate(spec.layers):
                q.append(self._synth(synth.STREAM_Q, l, reqs, pos, spec.Hq))
                k.append(self._synth(synth.STREAM_K, l, reqs, pos, hkv))
                v.append(self._synth(synth.STREAM_V, l, reqs, pos, hkv))
            seq_h = self.lens + s + 1
            steps.append(dict(q=q, k=k, v=v, seq_h=seq_h, pre_h=seq_h - 1,
                              seq_d=torch.tensor(seq_h, device=self.dev),
                              pre_d=torch.tensor(seq_h - 1, device=self.dev)))
        return steps

    def alloc_decode_buffers(self):
        spec = self.spec
        self.out_full = torch.empty(self.B, dtype=torch.int64, device=self.dev)
        self.out_swa = torch.empty(self.B, dtype=torch.int64, device=self.dev)
        self.plan = torch.zeros(api.swa_plan_bytes(self.ctx, self.B, 1), dtype=torch.uint8,
                                device=self.dev)
        # Decode steps pass their own longest request, anywhere from the
        # prompt length up to max_seq_len: size for the largest need over that
        # range (the split size, hence the split count, depends on it).
        kinds = {}
        for l, (kind, _, hkv) in enumerate(spec.layers):
            kinds.setdefault((kind, hkv), l)
        lo = max(1, int(self.seq0.max()) - 1)
        wsb = max(api.swa_attn_decode_ws_bytes(self.ctx, l, self.B, m)
                  for l in kinds.values()
                  for m in list(range(lo, self.max_seq_len + 1, 16)) + [self.max_seq_len])
        self.ws = torch.zeros(wsb, dtype=torch.uint8, device=self.dev)
        self.outs = [torch.empty((self.B, spec.Hq, spec.D), dtype=self.in_dtype, device=self.dev)
                     for _ in spec.layers]

    def decode_step(self, inp, attn_events=None, fused=True):
        """One decode step: evict (interval), alloc_decode, plan, then per layer
        store_kv + attn_decode - one swa_store_kv_attn_decode call when
        `fused`, else the two calls.  attn_events: optional dict layer ->
        (start, end) CUDA events recorded around that layer's attention."""
        spec = self.spec
        if self.trace is not None:
            self.trace.append(("evict", self.rows.tolist(), inp["pre_h"].tolist(),
                               self.evicted.tolist(), spec.interval))
        ev_before = self.evicted.copy()
        api.swa_evict_swa(self.ctx, self.rt, self.rows_d, inp["pre_d"], self.evicted_d,
                          inp["pre_h"], self.evicted, interval=spec.interval)
        launches = 3 if (self.evicted != ev_before).any() else 0
        if self.trace is not None:
            self.trace.append(("decode", self.rows.tolist(), inp["seq_h"].tolist()))
        api.swa_alloc_decode(self.ctx, inp["seq_d"], None, inp["seq_h"], self.out_full,
                             self.out_swa, req_to_token=self.rt, req_idx=self.rows_d)
        api.swa_plan(self.ctx, self.rt, self.rows_d, None, inp["seq_d"], self.plan, 1)
        # The longest request of this step (the workspace is sized for the
        # largest it can reach); the split size follows it.
        msl = int(inp["seq_h"].max())
        for l in range(len(spec.layers)):
            if not fused:
                api.swa_store_kv(self.ctx, l, inp["k"][l], inp["v"][l], self.out_full,
                                 self.out_swa)
            ev = attn_events.get(l) if attn_events else None
            if ev is not None:
                ev[0].record()
            if fused:
                api.swa_store_kv_attn_decode(self.ctx, l, self.rt, self.rows_d, inp["seq_d"], msl,
                                             self.plan, inp["q"][l], inp["k"][l], inp["v"][l],
                                             self.out_full, self.out_swa, self.sinks_d[l],
                                             self.scale, self.outs[l], self.ws)
            else:
                api.swa_attn_decode(self.ctx, l, self.rt, self.rows_d, inp["seq_d"], msl,
                                    self.plan, inp["q"][l], self.sinks_d[l], self.scale,
                                    self.outs[l], self.ws)
            if ev is not None:
                ev[1].record()
            launches += 1 if fused and api.swa_last_attn_path(self.ctx) == 1 else 2
        self.last_launches = launches + 2 + 1      # + alloc_decode, plan
        self.lens = inp["seq_h"].copy()

    # -- extend (one chunked-prefill round) -------------------------------------
    def make_extend_inputs(self, chunk: int):
        """Everything one chunk round of every request reads that is not the
        method's own state: the chunk's q/k/v of every layer (drawn on the
        device), lengths, query offsets, the plan buffer and the workspace."""
        spec = self.spec
        pre = self.lens.copy()
        seq = pre + chunk
        ext = seq - pre
        indptr = np.concatenate([[0], np.cumsum(ext)]).astype(np.int64)
        n = int(indptr[-1])
        d = lambda x: torch.tensor(x, device=self.dev)
        meta = dict(pre=pre, seq=seq, indptr=indptr, n=n, pre_d=d(pre), seq_d=d(seq),
                    indptr_d=d(indptr))
        meta["plan"] = torch.zeros(api.swa_plan_bytes(self.ctx, self.B, int(ext.max())),
                                   dtype=torch.uint8, device=self.dev)
        reqs = torch.tensor(np.repeat(self.rows, ext), device=self.dev)
        pos = torch.tensor(np.concatenate([np.arange(p, s) for p, s in zip(pre, seq)]),
                           device=self.dev)
        meta["q"] = [self._synth(synth.STREAM_Q, l, reqs, pos, spec.Hq)
                     for l in range(len(spec.layers))]
        meta["k"] = [self._synth(synth.STREAM_K, l, reqs, pos, h)
                     for l, (_, _, h) in enumerate(spec.layers)]
        meta["v"] = [self._synth(synth.STREAM_V, l, reqs, pos, h)
                     for l, (_, _, h) in enumerate(spec.layers)]
        meta["out"] = [torch.empty_like(x) for x in meta["q"]]
        meta["out_full"] = torch.empty(n, dtype=torch.int64, device=self.dev)
        meta["out_swa"] = torch.empty(n, dtype=torch.int64, device=self.dev)
        wsb = max(api.swa_attn_extend_ws_bytes(self.ctx, l, n, int(seq.max()))
                  for l in range(len(spec.layers)))
        meta["ws"] = torch.zeros(wsb, dtype=torch.uint8, device=self.dev)
        return meta

    def extend_round(self, chunk: int, attn_events=None, evict_events=None, meta=None):
        """One chunk of every request: eviction before the chunk, alloc_extend,
        KV store of every layer, the per-batch plan and extend attention on
        every layer, all on inputs prepared beforehand (``meta`` from
        make_extend_inputs, drawn here when not given).  Returns ``meta``
        with the outputs (kept for parity checks)."""
        spec = self.spec
        if meta is None:
            meta = self.make_extend_inputs(chunk)
        idx = np.arange(self.B)
        self._evict(idx, 0, evict_events)
        pre, seq = meta["pre"], meta["seq"]
        if self.trace is not None:
            self.trace.append(("extend", self.rows.tolist(), pre.tolist(), seq.tolist()))
        api.swa_alloc_extend(self.ctx, meta["pre_d"], meta["seq_d"], None, pre, seq,
                             meta["out_full"], meta["out_swa"], req_to_token=self.rt,
                             req_idx=self.rows_d)
        for l in range(len(spec.layers)):
            api.swa_store_kv(self.ctx, l, meta["k"][l], meta["v"][l], meta["out_full"],
                             meta["out_swa"])
        self.lens[idx] = seq
        ext_max = int((seq - pre).max())
        api.swa_plan(self.ctx, self.rt, self.rows_d, meta["pre_d"], meta["seq_d"], meta["plan"],
                     ext_max)
        self.extend_attention(meta, attn_events)
        return meta

    def extend_attention(self, meta, attn_events=None):
        spec = self.spec
        ext_max = int((meta["seq"] - meta["pre"]).max())
        for l in range(len(spec.layers)):
            ev = attn_events.get(l) if attn_events else None
            if ev is not None:
                ev[0].record()
            api.swa_attn_extend(self.ctx, l, self.rt, self.rows_d, meta["pre_d"], meta["seq_d"],
                                meta["indptr_d"], meta["n"], ext_max, int(meta["seq"].max()),
                                meta["plan"], meta["q"][l], self.sinks_d[l], self.scale,
                                meta["out"][l], meta["ws"])
            if ev is not None:
                ev[1].record()

    def extend_flops(self, meta) -> dict:
        """Algorithmic flops of extend attention: 4*D per attended (q-head, key)."""
        spec = self.spec
        full = swa = 0
        for kind, w, hkv in spec.layers:
            pairs = 0
            for p0, s in zip(meta["pre"], meta["seq"]):
                p = np.arange(p0, s)
                if kind == FULL:
                    n = p + 1
                elif kind == SLIDING:
                    n = p - np.maximum(0, p - w) + 1
                else:
                    n = p - (p // w) * w + 1
                pairs += int(n.sum())
            f = 4 * spec.D * spec.Hq * pairs
            if kind == FULL:
                full += f
            else:
                swa += f
        return {"full": full, "swa": swa, "total": full + swa}

    def launches_per_step(self) -> int:
        """Kernel launches of the last decode_step: eviction (3, only when a
        request evicts), alloc_decode (2), plan (1), and per layer the store and
        the attention (one launch when the tensor-core decode kernel stores the
        token itself)."""
        return self.last_launches

    def kv_bytes_per_step(self, seq_h=None) -> dict:
        """Algorithmic K+V bytes read by attention in one decode step."""
        spec = self.spec
        seq = self.lens + 1 if seq_h is None else seq_h
        es = ESIZE[spec.dtype]
        full = swa = 0
        for kind, w, hkv in spec.layers:
            p = seq - 1
            if kind == FULL:
                n = seq
            elif kind == SLIDING:
                n = p - np.maximum(0, p - w) + 1
            else:
                n = p - (p // w) * w + 1
            b = int(n.sum()) * hkv * spec.D * 2 * es
            if kind == FULL:
                full += b
            else:
                swa += b
        return {"full": full, "swa": swa, "total": full + swa}
