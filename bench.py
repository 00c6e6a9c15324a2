"""Benchmark of the hybrid sliding-window two-pool decode path on GB300.

One step = one decode step of the whole batch through the path: out-of-window
SWA eviction (interval 128), alloc_decode in both pools + mapping, the
per-batch SWA plan, then for every layer the KV store of the new token and
paged attention (sliding layers through the SWA pool, full layers through
req_to_token).  Inputs (q/k/v of the step, the KV cache built by a chunked
prefill of the same method) are resident in HBM before timing; the KV read
per step (~23 GB for the MiMo-shaped workload) is far larger than L2, so no
flush is needed between steps.

value  = algorithmic K+V bytes attended per step / device time per step (GB/s)
e2e    = the same bytes / time per step when each step also copies its q/k/v
         from pinned host memory and copies every layer's output back.
roofline = the full-layer attention kernel alone (the dominant kernel), timed
         with CUDA events around each of its launches.

The default (MiMo-shaped) line also carries: a steady-state run long enough
that every request crosses the eviction interval (eviction cost amortised);
the GPT-OSS- and Llama4-shaped decode workloads at full size; the Tiny
configuration's per-step latency; the chunked-prefill extend (attention
TFLOP/s, and the whole round: eviction, allocation, store, plan, attention);
eviction slots/s; and the CPU oracle timed on the host's cores (one core and
all cores, whole decode steps; extend extrapolated by flops).

``--impl reference`` times the CPU oracle on a bounded sample of the same
workload instead (single-threaded numpy, float64).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% HBM peak) and tokens/s; extend TFLOP/s; evict slots/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------- CPU oracle ---
def cpu_model():
    """Host CPU model name and core count (for the baseline's record)."""
    name = vendor = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and name is None:
                name = v.strip()
            if k.strip() == "Vendor ID" and vendor is None:
                vendor = v.strip()
    except Exception:
        pass
    return name or vendor or "unknown", os.cpu_count() or 1


def oracle_request_step(workload, b):
    """The oracle's whole decode step for request b of the workload: eviction
    pass (the workload's interval) and alloc_decode on an oracle allocator
    holding the request's replayed chunked prefill, then for every layer the
    window translation through req_to_token and the mapping, the store
    encoding of the new token's K/V rows, and the brute-force attention of all
    query heads.  K/V values come from the seeded generator, drawn once per
    (request, layer shape) and used by every layer of that shape (the
    oracle's work does not depend on the values); drawing is not timed.
    Returns (oracle seconds by phase, attended K+V bytes)."""
    import numpy as np
    from hybrid_sliding_window_gb300 import synth
    from hybrid_sliding_window_gb300.workloads import ESIZE, FULL, SPECS
    from oracle import allocator as OA
    from oracle import attention as OT
    from oracle import codecs as OC
    spec = SPECS[workload]
    ps, lb = spec.ps, spec.lookback()
    seq = int(spec.seq_lens()[b])          # the decode step's length (new token included)
    row = b + 1
    okind = {0: OT.FULL, 1: OT.SLIDING, 2: OT.CHUNKED}
    nf = (-(-(seq + ps) // ps) + 2) * ps
    ns = (-(-(spec.chunk + lb + spec.interval) // ps) + 4) * ps
    oa = OA.TwoPoolAllocator(nf, ns, ps)
    ort = np.zeros((row + 1, seq + ps), np.int64)
    pre, ev = 0, [0]
    while pre < seq - 1:                   # replayed prefill (setup, not timed)
        ev, _ = OA.evict_swa(oa, ort, [row], [pre], ev, [0], lb, 0)
        new = min(pre + spec.chunk, seq - 1)
        last = [int(ort[row, pre - 1]) if pre else -1]
        full, _ = oa.alloc_extend([pre], [new], last)
        ort[row, pre:new] = full
        pre = new
    ev, _ = OA.evict_swa(oa, ort, [row], [pre], ev, [0], lb, 0)
    ph = dict(evict_alloc=0.0, plan=0.0, store=0.0, attention=0.0)
    t0 = time.perf_counter()
    ev, _ = OA.evict_swa(oa, ort, [row], [seq - 1], ev, [0], lb, spec.interval)
    full, _ = oa.alloc_decode([seq], [int(ort[row, seq - 2])])
    ort[row, seq - 1] = full[0]
    ph["evict_alloc"] += time.perf_counter() - t0
    p = seq - 1
    drawn = {}
    nbytes = 0
    bf = spec.dtype != "f32"
    for l, (kind, w, hkv) in enumerate(spec.layers):
        J = list(OT.key_positions(okind[kind], w, p))
        key = (kind, w, hkv)
        if key not in drawn:
            K = synth.tokens(spec.seed, synth.STREAM_K, l, [row] * len(J), J, hkv, spec.D, bf16=bf)
            V = synth.tokens(spec.seed, synth.STREAM_V, l, [row] * len(J), J, hkv, spec.D, bf16=bf)
            if spec.dtype == "e4m3":
                K = OC.e4m3_decode(OC.e4m3_encode(K))
                V = OC.e4m3_decode(OC.e4m3_encode(V))
            drawn[key] = (K.astype(np.float64), V.astype(np.float64))
        K, V = drawn[key]
        q = synth.tokens(spec.seed, synth.STREAM_Q, l, [row], [p], spec.Hq, spec.D, bf16=bf)[0]
        sinks = synth.sinks(spec.seed, l, spec.Hq) if spec.sinks else None
        t0 = time.perf_counter()
        slots = [int(ort[row, j]) for j in J]
        if kind != FULL:
            slots = [oa.mapping[s] for s in slots]
            assert all(s > 0 for s in slots)
        t1 = time.perf_counter()
        enc = OC.e4m3_encode if spec.dtype == "e4m3" else (OC.bf16_encode if bf else np.float32)
        enc(K[-1].astype(np.float32))
        enc(V[-1].astype(np.float32))
        t2 = time.perf_counter()
        OT.attend_heads(q, K, V, sinks, 1.0 / np.sqrt(spec.D))
        t3 = time.perf_counter()
        ph["plan"] += t1 - t0
        ph["store"] += t2 - t1
        ph["attention"] += t3 - t2
        nbytes += len(J) * hkv * spec.D * 2 * ESIZE[spec.dtype]
    return ph, nbytes, os.getpid()


def _oracle_request_job(a):
    return oracle_request_step(*a)


def oracle_extend_sample(n_full=12, n_swa=128):
    """The oracle's extend attention on sampled chunk queries of one request
    of the chunked-prefill workload (24576-token prefix + 8192 chunk): n_full
    queries of a full layer and n_swa of a sliding layer, all query heads.
    Returns per layer kind (flops, seconds)."""
    import numpy as np
    from hybrid_sliding_window_gb300 import synth
    from hybrid_sliding_window_gb300.workloads import EXTEND_CHUNK, EXTEND_PREFIX, EXTEND_SPEC, FULL
    from oracle import attention as OT
    spec = EXTEND_SPEC
    rng = np.random.default_rng(0)
    out = {}
    for l, n in ((4, n_full), (0, n_swa)):
        kind, w, hkv = spec.layers[l]
        okind = OT.FULL if kind == FULL else OT.SLIDING
        pos = sorted(EXTEND_PREFIX + int(i) for i in rng.integers(0, EXTEND_CHUNK, n))
        lo = min(OT.key_positions(okind, w, p).start for p in pos)
        J = np.arange(lo, pos[-1] + 1)
        K = synth.tokens(spec.seed, synth.STREAM_K, l, [1] * len(J), J, hkv, spec.D).astype(np.float64)
        V = synth.tokens(spec.seed, synth.STREAM_V, l, [1] * len(J), J, hkv, spec.D).astype(np.float64)
        sinks = synth.sinks(spec.seed, l, spec.Hq)
        secs, flops = 0.0, 0
        for p in pos:
            r = OT.key_positions(okind, w, p)
            q = synth.tokens(spec.seed, synth.STREAM_Q, l, [1], [p], spec.Hq, spec.D)[0]
            t0 = time.perf_counter()
            OT.attend_heads(q, K[r.start - lo:r.stop - lo], V[r.start - lo:r.stop - lo], sinks,
                            1.0 / np.sqrt(spec.D))
            secs += time.perf_counter() - t0
            flops += 4 * spec.D * spec.Hq * len(r)
        out["full" if kind == FULL else "swa"] = (flops, secs)
    return out


def _pin_blas():
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"


def cpu_child(workload, budget_s, all_cores, extend):
    """Body of the CPU-baseline child process (no GPU visible): prints one
    JSON line."""
    import multiprocessing as mp
    import numpy as np
    from hybrid_sliding_window_gb300.workloads import SPECS
    spec = SPECS[workload]
    order = [int(i) for i in np.random.default_rng(7).permutation(spec.batch)]
    # single core: whole requests' steps until the oracle time reaches the budget
    tot = dict(evict_alloc=0.0, plan=0.0, store=0.0, attention=0.0)
    nbytes, done = 0, []
    for b in order:
        ph, nb, _ = oracle_request_step(workload, b)
        for k in tot:
            tot[k] += ph[k]
        nbytes += nb
        done.append(b)
        if sum(tot.values()) >= budget_s:
            break
    secs = sum(tot.values())
    res = {"value": nbytes / secs / 1e9, "seconds": secs, "bytes": nbytes, "requests": len(done),
           "phases_s": {k: round(v, 3) for k, v in tot.items()}}
    if all_cores:
        n = os.cpu_count() or 1
        reqs = (order * ((n * 2) // len(order) + 1))[:max(len(done), 2 * n)]
        with mp.get_context("spawn").Pool(n, initializer=_pin_blas) as pool:
            per = {}
            bsum = 0
            for ph, nb, pid in pool.imap_unordered(_oracle_request_job,
                                                   [(workload, b) for b in reqs]):
                per[pid] = per.get(pid, 0.0) + sum(ph.values())
                bsum += nb
        busiest = max(per.values())
        res["all_cores"] = {"value": bsum / busiest / 1e9, "cores": len(per), "requests": len(reqs),
                            "bytes": bsum, "busiest_worker_s": busiest}
    if extend:
        res["extend"] = oracle_extend_sample()
    print(json.dumps(res))


def cpu_baseline(workload, budget_s, all_cores=True, extend=True):
    """The oracle, as it stands, timed on the host's cores in a child process
    with BLAS pinned to one thread per process and no GPU visible."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
            f"bench.cpu_child({workload!r}, {budget_s!r}, {all_cores!r}, {extend!r})")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=900)
    if r.returncode != 0:
        raise RuntimeError("cpu baseline failed: " + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    from hybrid_sliding_window_gb300.workloads import SPECS
    spec = SPECS[workload]
    model, ncpu = cpu_model()
    out = {"value": round(d["value"], 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "cpu": model, "nproc": ncpu,
           "sample": (f"whole decode steps of {d['requests']} of the {spec.batch} requests (eviction "
                      f"pass, alloc_decode, window translation, KV store encoding and attention of "
                      f"all {spec.Hq} query heads on every one of the {len(spec.layers)} layers): "
                      f"{d['bytes'] / 1e9:.2f} GB of attended K+V in {d['seconds']:.1f} s of "
                      f"float64 numpy oracle time on one host core"),
           "phases_s": d["phases_s"]}
    if "all_cores" in d:
        a = d["all_cores"]
        out["all_cores"] = {"value": round(a["value"], 4), "unit": "GB/s", "cores": a["cores"],
                            "sample": f"{a['requests']} request steps spread over {a['cores']} "
                                      f"processes; time = the busiest process's oracle time"}
    if "extend" in d:
        from hybrid_sliding_window_gb300.workloads import EXTEND_SPEC
        f_full, s_full = d["extend"]["full"]
        f_swa, s_swa = d["extend"]["swa"]
        out["extend"] = {
            "value": round((f_full + f_swa) / (s_full + s_swa) / 1e12, 6), "unit": "TFLOP/s",
            "cores": 1, "kind": "oracle, extrapolated",
            "extrapolated_round_s": None,
            "sample": "sampled chunk queries of one request of the chunked-prefill workload, all "
                      "64 query heads: a full layer and a sliding layer; a whole round's time "
                      "extrapolated by the algorithmic flops of each layer kind"}
        # Algorithmic flops of one round: 4 * D per (query head, attended key).
        import numpy as np
        from hybrid_sliding_window_gb300.workloads import EXTEND_CHUNK, EXTEND_PREFIX, FULL
        p = np.arange(EXTEND_PREFIX, EXTEND_PREFIX + EXTEND_CHUNK, dtype=np.float64)
        per_pair = 4 * EXTEND_SPEC.D * EXTEND_SPEC.Hq * EXTEND_SPEC.batch
        rf = rs = 0.0
        for kind, w, _ in EXTEND_SPEC.layers:
            if kind == FULL:
                rf += per_pair * (p + 1).sum()
            else:
                rs += per_pair * (np.minimum(p, w) + 1).sum()
        out["extend"]["extrapolated_round_s"] = round(rf / (f_full / s_full)
                                                      + rs / (f_swa / s_swa), 1)
        out["extend"]["round_flops"] = rf + rs
    return out


# ------------------------------------------------------------------ clocks ---
class ClockSampler:
    def __init__(self, index=0):
        self.proc = None
        self.path = None
        self.index = index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader",
                                          "-lms", "200", "-i", str(self.index)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        def mhz(s):
            try:
                return float(s.split()[0])
            except Exception:
                return None
        sm = [mhz(r[1]) for r in rows if mhz(r[1]) is not None]
        mx = [mhz(r[2]) for r in rows if mhz(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- native ---
def spec_for(args, name):
    from hybrid_sliding_window_gb300.workloads import SPECS
    spec = SPECS[name]
    if args.batch or args.layers or args.r or args.chunk:
        # Reduced shapes for profiler captures only (named in the config line).
        import dataclasses
        spec = dataclasses.replace(
            spec, batch=args.batch or spec.batch,
            layers=spec.layers[:args.layers] if args.layers else spec.layers,
            r=args.r or spec.r, chunk=args.chunk or spec.chunk,
            description=spec.description + f" [reduced: batch={args.batch or spec.batch}, "
                                           f"layers={args.layers or len(spec.layers)}, "
                                           f"r={args.r or spec.r}, chunk={args.chunk or spec.chunk}]")
    return spec


def decode_timed(st, inputs, W, K, fused=True, barrier=None, index=0):
    """W untimed decode steps, then K steps timed with CUDA events on the
    launching stream (plus per-launch events around every full layer's
    attention).  Returns the step time, the full-layer launch time, the
    algorithmic bytes and the launch count."""
    import torch
    from hybrid_sliding_window_gb300.workloads import FULL
    spec = st.spec
    for s in range(W):
        st.decode_step(inputs[s], fused=fused)
    full_layers = [l for l, (k, _, _) in enumerate(spec.layers) if k == FULL]
    ev = {l: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)] for l in full_layers}
    bytes_steps, attn_bytes, launches = [], [], 0
    (barrier or torch.cuda.synchronize)()
    clk = ClockSampler(index)
    clk.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(K):
        inp = inputs[W + s]
        b = st.kv_bytes_per_step(inp["seq_h"])
        bytes_steps.append(b["total"])
        attn_bytes.append(b["full"] / len(full_layers))
        st.decode_step(inp, {l: ev[l][s] for l in full_layers}, fused=fused)
        launches += st.launches_per_step()
    e1.record()
    (barrier or torch.cuda.synchronize)()
    clocks = clk.stop()
    durs = [ev[l][s][0].elapsed_time(ev[l][s][1]) for l in full_layers for s in range(K)]
    return dict(t_ms=e0.elapsed_time(e1), full_ms=sum(durs) / len(durs), bytes=sum(bytes_steps),
                bytes_per_step=sum(bytes_steps) / K, attn_bytes=sum(attn_bytes) / len(attn_bytes),
                launches=launches, clocks=clocks)


def decode_summary(spec, r, K, workload):
    """The decode figures of one workload: GB/s of attended K+V, tokens/s and
    the dominant (full-layer) kernel against the measured copy peak."""
    peak, peak_kind = peaks()
    value = r["bytes"] / (r["t_ms"] / 1e3) / 1e9
    ach = r["attn_bytes"] / (r["full_ms"] / 1e3) / 1e9
    return {
        "value": round(value, 2), "unit": "GB/s", "hbm_frac": round(value / peak, 4),
        "ms_per_step": round(r["t_ms"] / K, 4), "steps": K,
        "tokens_per_s": round(spec.batch * K / (r["t_ms"] / 1e3), 1),
        "kv_bytes_per_step": int(r["bytes_per_step"]),
        "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(ach / peak, 4),
                     "traffic": stored_traffic(f"{workload}_decode_traffic.json", DECODE_SOURCES),
                     "kernel": "swa_store_kv_attn_decode on full layers (k_decode_mma)",
                     "peak_source": peak_kind, "avg_launch_ms": round(r["full_ms"], 4)},
        "clocks": r["clocks"], "gpu_launches": r["launches"],
    }


def steady_state(st, n_steps, fused=True):
    """n_steps more decode steps timed as one region, long enough that every
    request crosses the eviction interval: the eviction passes run inside the
    timed steps, so their cost is amortised into this figure."""
    import torch
    inputs = st.make_decode_inputs(n_steps)
    ev0 = st.evicted.copy()
    passes, nbytes = 0, 0
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for inp in inputs:
        before = st.evicted.copy()
        nbytes += st.kv_bytes_per_step(inp["seq_h"])["total"]
        st.decode_step(inp, fused=fused)
        passes += int((st.evicted != before).any())
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    peak, _ = peaks()
    return {"steps": n_steps, "value": round(nbytes / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "hbm_frac": round(nbytes / (ms / 1e3) / 1e9 / peak, 4),
            "ms_per_step": round(ms / n_steps, 4), "steps_with_eviction": passes,
            "requests_evicting": int((st.evicted != ev0).sum()),
            "evicted_slots": int((st.evicted - ev0).sum())}


def graph_steps(st, n_steps, fused=True):
    """n_steps decode steps captured into one CUDA graph, replayed once and
    timed with CUDA events: the steps' device time without host launch
    gaps.  The host-side bookkeeping (lengths, eviction decisions, the
    library's free-count mirrors) runs during capture and the single replay
    executes each captured step once, so host and device state stay in step."""
    import torch
    inputs = st.make_decode_inputs(n_steps)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    nbytes, passes, launches = 0, 0, 0
    with torch.cuda.graph(g):
        for inp in inputs:
            before = st.evicted.copy()
            nbytes += st.kv_bytes_per_step(inp["seq_h"])["total"]
            st.decode_step(inp, fused=fused)
            passes += int((st.evicted != before).any())
            launches += st.launches_per_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    del g
    peak, _ = peaks()
    return {"steps": n_steps, "value": round(nbytes / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "hbm_frac": round(nbytes / (ms / 1e3) / 1e9 / peak, 4),
            "ms_per_step": round(ms / n_steps, 4), "us_per_step": round(ms * 1e3 / n_steps, 2),
            "steps_with_eviction": passes, "gpu_launches": launches}


def decode_sub(args, name, K, W):
    """A whole decode workload (build, warm-up, K timed steps) for the line's
    per-workload objects; its state is freed before returning."""
    import gc
    import torch
    from hybrid_sliding_window_gb300.workloads import DecodeState
    spec = spec_for(args, name)
    st = DecodeState(spec, max_steps=W + K + 4)
    st.prefill()
    st.alloc_decode_buffers()
    inputs = st.make_decode_inputs(W + K)
    r = decode_timed(st, inputs, W, K, index=int(os.environ.get("LOCAL_RANK", "0")))
    out = decode_summary(spec, r, K, name)
    out["workload"] = spec.description
    del st, inputs
    gc.collect()
    torch.cuda.empty_cache()
    return out


def tiny_latency(args, K=64, W=8):
    """The Tiny configuration: per-step device time of whole decode steps
    (eviction every 8 slid-out tokens, allocation, plan, store and attention
    of both layers), each step bracketed by its own CUDA events."""
    import gc
    import statistics as stt
    import torch
    from hybrid_sliding_window_gb300 import api
    from hybrid_sliding_window_gb300.workloads import SPECS, DecodeState
    spec = SPECS["tiny"]
    st = DecodeState(spec, max_steps=W + 2 * K + 4)
    st.prefill()
    st.alloc_decode_buffers()
    inputs = st.make_decode_inputs(W + K)
    for s in range(W):
        st.decode_step(inputs[s])
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    passes, launches = 0, 0
    torch.cuda.synchronize()
    for s in range(K):
        before = st.evicted.copy()
        evs[s][0].record()
        st.decode_step(inputs[W + s])
        evs[s][1].record()
        passes += int((st.evicted != before).any())
        launches += st.launches_per_step()
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    assert api.swa_device_check(st.ctx) == 0
    out = {"workload": spec.description, "unit": "us per decode step", "steps": K,
           "median_us": round(stt.median(us), 2), "p90_us": round(us[int(0.9 * (K - 1))], 2),
           "min_us": round(us[0], 2), "steps_with_eviction": passes,
           "launches_per_step": round(launches / K, 2),
           "kv_bytes_per_step": int(st.kv_bytes_per_step()["total"]),
           "timing": "CUDA events around each step issued from Python (includes the host's "
                     "launch gaps)"}
    try:
        gr = graph_steps(st, K)
        assert api.swa_device_check(st.ctx) == 0
        out["graph"] = {"us_per_step": gr["us_per_step"], "steps": K,
                        "steps_with_eviction": gr["steps_with_eviction"],
                        "timing": f"{K} steps captured in one CUDA graph, replayed once"}
    except Exception as e:   # the eager figure stands; say why the graph one is missing
        out["graph"] = {"error": str(e)[:300]}
    del st, inputs
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_native(args, rank, world):
    import numpy as np
    import torch
    from hybrid_sliding_window_gb300 import api
    from hybrid_sliding_window_gb300.workloads import DecodeState

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    api.lib()
    spec = spec_for(args, args.workload)
    W, K = args.warmup, args.steps
    # Step headroom: the timed and e2e steps, the steady-state run, and one
    # speculative step's drafts (<= 1024).
    steady_n = args.steady_steps
    st = DecodeState(spec, max_steps=W + 2 * K + steady_n + args.graph_steps + 4 + 1024,
                     swa_ring=args.swa_ring)
    if args.attn_path != -1:
        api.swa_set_attn_path(st.ctx, args.attn_path)
    t0 = time.time()
    st.prefill()
    setup_s = time.time() - t0
    st.alloc_decode_buffers()
    inputs = st.make_decode_inputs(W + 2 * K)
    torch.cuda.synchronize()
    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()

    r = decode_timed(st, inputs, W, K, fused=not args.separate_store, barrier=barrier, index=local)
    t_ms, launches, clocks = r["t_ms"], r["launches"], r["clocks"]
    assert api.swa_device_check(st.ctx) == 0, "device-side check flagged an error"
    # e2e: the same steps fed from pinned host memory, outputs copied back.
    # A step's inputs (q, k, v of every layer and the lengths) travel as one
    # pinned buffer and one copy, the outputs of every layer come back as one
    # copy; the copies run on their own stream with double-buffered device
    # buffers, so step s+1's inputs and step s's outputs move while the GPU
    # computes step s.
    B = st.B
    parts = [(key, l) for key in ("q", "k", "v") for l in range(len(inputs[0][key]))]
    layout, off = {}, 0
    for key, l in parts:
        t = inputs[0][key][l]
        layout[(key, l)] = (off, tuple(t.shape), t.dtype, t.numel() * t.element_size())
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    for key in ("seq", "pre"):
        layout[key] = off
        off += (B * 8 + 255) // 256 * 256
    in_bytes = off

    def in_views(buf):
        d = {"q": [], "k": [], "v": []}
        for key, l in parts:
            o, shape, dt, n = layout[(key, l)]
            d[key].append(buf[o:o + n].view(dt).view(shape))
        for key in ("seq", "pre"):
            d[key] = buf[layout[key]:layout[key] + B * 8].view(torch.int64)
        return d

    host_in = []
    for s in range(K):
        src = inputs[W + K + s]
        hb = torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True)
        hv = in_views(hb)
        for key, l in parts:
            hv[key][l].copy_(src[key][l].cpu())
        hv["seq"].copy_(torch.from_numpy(np.asarray(src["seq_h"], np.int64)))
        hv["pre"].copy_(torch.from_numpy(np.asarray(src["pre_h"], np.int64)))
        host_in.append(hb)
    dev_buf = [torch.empty(in_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    dev_in = [in_views(b) for b in dev_buf]
    o_sizes = [o.numel() * o.element_size() for o in st.outs]
    out_bytes = sum(o_sizes)
    out_flat = [torch.empty(out_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    out_sets = []
    for fb in out_flat:
        views, o = [], 0
        for t, n in zip(st.outs, o_sizes):
            views.append(fb[o:o + n].view(t.dtype).view(t.shape))
            o += n
        out_sets.append(views)
    host_out = [torch.empty(out_bytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    h2d, d2h = in_bytes, out_bytes
    outs_saved = st.outs
    cs = torch.cuda.current_stream()
    ps = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    e2e_bytes = 0
    barrier()
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    x0.record(cs)
    ps.wait_event(x0)
    with torch.cuda.stream(ps):
        dev_buf[0].copy_(host_in[0], non_blocking=True)
        in_ready[0].record(ps)
    for s in range(K):
        i = s % 2
        if s + 1 < K:                      # next step's inputs, behind this step's compute
            j = (s + 1) % 2
            with torch.cuda.stream(ps):
                if s >= 1:
                    ps.wait_event(in_free[j])
                dev_buf[j].copy_(host_in[s + 1], non_blocking=True)
                in_ready[j].record(ps)
        cs.wait_event(in_ready[i])
        if s >= 2:
            cs.wait_event(out_free[i])     # step s-2's outputs have left this buffer
        src = inputs[W + K + s]
        d = dev_in[i]
        st.outs = out_sets[i]
        e2e_bytes += st.kv_bytes_per_step(src["seq_h"])["total"]
        st.decode_step(dict(q=d["q"], k=d["k"], v=d["v"], seq_h=src["seq_h"], pre_h=src["pre_h"],
                            seq_d=d["seq"], pre_d=d["pre"]), fused=not args.separate_store)
        in_free[i].record(cs)
        out_ready[i].record(cs)
        with torch.cuda.stream(ps):
            ps.wait_event(out_ready[i])
            host_out[i].copy_(out_flat[i], non_blocking=True)
            out_free[i].record(ps)
    cs.wait_stream(ps)
    x1.record(cs)
    barrier()
    st.outs = outs_saved
    e2e_ms = x0.elapsed_time(x1)
    assert api.swa_device_check(st.ctx) == 0
    spec_alloc = spec_alloc_rate(st) if rank == 0 else None
    kernel_ids = translate_rate(st) if rank == 0 else None

    steady = steady_state(st, steady_n, fused=not args.separate_store) if steady_n else None
    assert api.swa_device_check(st.ctx) == 0
    graph = None
    if args.graph_steps and world == 1:
        try:
            graph = graph_steps(st, args.graph_steps, fused=not args.separate_store)
            assert api.swa_device_check(st.ctx) == 0
        except Exception as e:   # the eager figures stand; say why this one is missing
            graph = {"error": str(e)[:300]}

    (t_ms_max, e2e_max), (tot_bytes, tot_e2e) = reduce_ranks(
        [t_ms, e2e_ms], [float(r["bytes"]), float(e2e_bytes)], "cuda")
    if rank != 0:
        return None
    r["t_ms"], r["bytes"] = t_ms_max, tot_bytes
    summ = decode_summary(spec, dict(r, bytes_per_step=r["bytes_per_step"]), K, args.workload)
    summ["tokens_per_s"] = round(spec.batch * world * K / (t_ms_max / 1e3), 1)
    line = {
        "metric": METRIC, "value": summ["value"], "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(t_ms_max / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic",
        "config": {"workload": spec.description, "batch_per_gpu": spec.batch,
                   "kv_bytes_per_step": int(r["bytes_per_step"]),
                   "l2": "no flush: each step reads far more KV than the 129 MB L2",
                   "pools_tokens": {"full": st.size_full, "swa": st.size_swa},
                   "kv_store": ("separate swa_store_kv launch" if args.separate_store
                                else "inside the attention launch (swa_store_kv_attn_decode)"),
                   "swa_pool": (f"per-request ring of {st.ring_size} tokens" if st.swa_ring
                                else "paged"),
                   "setup_s": round(setup_s, 1)},
        "hbm_frac": summ["hbm_frac"],
        "tokens_per_s": summ["tokens_per_s"],
        "roofline": summ["roofline"],
        "e2e": {"value": round(tot_e2e / (e2e_max / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "per step one pinned host-to-device copy of q/k/v and lengths, one "
                          "device-to-host copy of all outputs, on a copy stream overlapped with "
                          "the previous / next step's compute"},
        "clocks": clocks,
        "gpu_launches": launches,
        "attn_path": api.swa_last_attn_path(st.ctx),
        "steady_state_with_eviction": steady,
        "cuda_graph": graph,
        "spec_alloc": spec_alloc,
        "translate_for_kernel": kernel_ids,
    }
    del st, inputs, host_in, dev_in, host_out
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    if world == 1 and not args.no_others and args.workload == "mimo" and not (
            args.batch or args.layers or args.r or args.chunk):
        # The other decode configurations, each at its full size (fewer
        # steps: every step reads 18-61 GB), and the Tiny configuration's
        # per-step latency.
        for name in ("gptoss", "llama4"):
            line[name] = decode_sub(args, name, K=max(5, min(K, 10)), W=3)
        line["tiny"] = tiny_latency(args)
    if world == 1 and not args.no_extend:
        # The other two figures the metric names: extend TFLOP/s and evict
        # slots/s, on the chunked-prefill workload (decode pools freed first).
        sub = argparse.Namespace(**vars(args))
        sub.steps, sub.warmup, sub.layers = 2, 1, 0
        ext = run_extend(sub, rank, world)
        line["extend"] = {k: ext[k] for k in ("value", "unit", "ms_per_step",
                                              "frac_of_sustained_bf16", "roofline", "clocks",
                                              "whole_round")}
        line["extend"]["workload"] = ext["config"]["workload"]
        line["evict"] = ext["evict"]
    if world == 1 and not args.no_cpu:
        try:
            line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds,
                                                extend=not args.no_extend)
        except Exception as e:  # the GPU number stands; say why the baseline is missing
            line["cpu_baseline"] = {"error": str(e)[:300]}
    return line


def reduce_ranks(max_vals, sum_vals, device):
    """Max of the times and sum of the work over ranks (any torch.distributed
    backend); identity on a single process."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return list(max_vals), list(sum_vals)
    mx = torch.tensor(list(max_vals), dtype=torch.float64, device=device)
    sm = torch.tensor(list(sum_vals), dtype=torch.float64, device=device)
    tdist.all_reduce(mx, op=tdist.ReduceOp.MAX)
    tdist.all_reduce(sm, op=tdist.ReduceOp.SUM)
    return mx.tolist(), sm.tolist()


def bf16_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def run_extend(args, rank, world, quiet=False):
    """Chunked-prefill extend, MiMo layers, 4 requests: a warm-up round
    (prefix 16384 -> 24576), then the configuration's round (24576-token
    prefix + 8192-token chunk) timed whole - eviction below the window,
    alloc_extend, the KV store of all 48 layers, the plan and the attention
    of all 48 layers - on inputs drawn beforehand; then the attention of that
    round repeated, with the full layers' launches timed one by one."""
    import gc
    import numpy as np
    import torch
    from hybrid_sliding_window_gb300 import api
    from hybrid_sliding_window_gb300.workloads import (EXTEND_CHUNK, EXTEND_PREFIX, EXTEND_SPEC,
                                                       DecodeState, FULL)
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    api.lib()
    spec = EXTEND_SPEC
    if args.layers:
        # Reduced layer count for profiler captures only (named in the config line).
        import dataclasses
        spec = dataclasses.replace(spec, layers=spec.layers[:args.layers],
                                   description=spec.description + f" [reduced: layers={args.layers}]")
    st = DecodeState(spec, max_steps=2 * EXTEND_CHUNK + 64)
    st.prefill(prompt=np.full(spec.batch, EXTEND_PREFIX - EXTEND_CHUNK, np.int64),
               final_evict=False)
    warm = st.make_extend_inputs(EXTEND_CHUNK)
    st.extend_round(EXTEND_CHUNK, meta=warm)
    del warm
    gc.collect()
    torch.cuda.empty_cache()
    full_layers = [l for l, (k, _, _) in enumerate(spec.layers) if k == FULL]
    meta = st.make_extend_inputs(EXTEND_CHUNK)
    ev_evict = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    slots_before = st.evicted.copy()
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    r0.record()
    st.extend_round(EXTEND_CHUNK, evict_events=ev_evict, meta=meta)
    r1.record()
    torch.cuda.synchronize()
    assert api.swa_device_check(st.ctx) == 0
    round_ms = r0.elapsed_time(r1)
    evict_ms = ev_evict[0].elapsed_time(ev_evict[1])
    evicted_slots = int((st.evicted - slots_before).sum())
    flops = st.extend_flops(meta)
    # Timed: the attention of the whole chunk round (all 48 layers), repeated.
    W, K = args.warmup, args.steps
    for _ in range(W):
        st.extend_attention(meta)
    evs = {l: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)] for l in full_layers}
    clk = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.synchronize()
    clk.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(K):
        st.extend_attention(meta, {l: evs[l][k] for l in full_layers})
    e1.record()
    torch.cuda.synchronize()
    clocks = clk.stop()
    t_ms = e0.elapsed_time(e1) / K
    full_ms = sum(evs[l][k][0].elapsed_time(evs[l][k][1]) for l in full_layers
                  for k in range(K)) / (K * len(full_layers))
    assert api.swa_device_check(st.ctx) == 0
    burst, sustained, src = bf16_peaks()
    per_full = flops["full"] / len(full_layers)
    ach = per_full / (full_ms / 1e3) / 1e12
    n_tok = int(meta["n"])
    return {
        "metric": METRIC, "value": round(flops["total"] / (t_ms / 1e3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(t_ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic",
        "config": {"workload": spec.description, "flops_per_round": flops["total"],
                   "l2": "no flush: each round reads ~1.3 GB of KV per full layer pass"},
        "frac_of_sustained_bf16": round(flops["total"] / (t_ms / 1e3) / 1e12 / sustained, 4),
        # The full layers are timed inside the repeated rounds (hundreds of
        # milliseconds of back-to-back tensor work, at the power cap): the
        # sustained bf16 peak is their denominator; the burst one is shown too.
        "roofline": {"bound": "tensor", "achieved": round(ach, 1), "peak": sustained,
                     "unit": "TFLOP/s", "frac": round(ach / sustained, 4),
                     "traffic": stored_traffic("extend_traffic.json", EXTEND_SOURCES),
                     "kernel": "swa_attn_extend on full layers (tcgen05)",
                     "peak_source": src + " bf16, sustained (timed inside a long step)",
                     "burst_peak": burst, "frac_of_burst": round(ach / burst, 4),
                     "avg_launch_ms": round(full_ms, 3)},
        "whole_round": {"ms": round(round_ms, 3),
                        "value": round(flops["total"] / (round_ms / 1e3) / 1e12, 2),
                        "unit": "TFLOP/s",
                        "steps": "eviction below the window, alloc_extend of 4 x 8192 tokens, "
                                 "the KV store of 48 layers, the plan and the attention of 48 "
                                 "layers, one round after a warm-up round",
                        "tokens": n_tok, "gpu_launches": 3 + 2 + 1 + 2 * len(spec.layers)},
        "evict": {"slots": evicted_slots, "ms": round(evict_ms, 4),
                  "slots_per_s": round(evicted_slots / (evict_ms / 1e3), 1)},
        "clocks": clocks, "attn_path": api.swa_last_attn_path(st.ctx),
        "gpu_launches": len(spec.layers) * K,
    }


def radix_requests(n_req, seed):
    """Synthetic prefix-cache traffic: requests = one of 16 shared 2048-token
    prompts + 1024 own tokens (page 64), drawn up front."""
    import numpy as np
    rng = np.random.default_rng(seed)
    prompts = rng.integers(1, 32000, size=(16, 2048), dtype=np.int32)
    return [np.concatenate([prompts[rng.integers(16)],
                            rng.integers(1, 32000, size=1024, dtype=np.int32)])
            for _ in range(n_req)]


def radix_ops(tree, reqs, evict_every=8):
    """Each request matches, locks, is 'prefilled' (its own tokens get fresh
    slots, the first 40 % of them slid out of the window), unlocks and is
    inserted; every few requests the cache is trimmed by SWA then full
    eviction.  Returns (ops, tokens)."""
    import numpy as np
    slot, ops, toks = 10 ** 6, 0, 0
    is_oracle = hasattr(tree, "take_releases")
    for i, t in enumerate(reqs):
        if is_oracle:
            t = t.tolist()
            e, slots, node = tree.match(t)
        else:
            e, slots, node = tree.match(t, as_numpy=True)
        span = tree.lock(node) if e else 0
        own = np.arange(slot, slot + len(t) - e, dtype=np.int64)
        slot += len(own)
        ev = ((e + int(0.4 * (len(t) - e))) // 64) * 64
        if e:
            tree.unlock(node, span)
        if is_oracle:
            tree.insert(t, list(slots) + own.tolist(), ev)
        else:
            tree.insert(t, np.concatenate([slots, own]), ev)
        ops += 2
        toks += 2 * len(t)
        if i % evict_every == evict_every - 1:
            if is_oracle:
                tree.evict_swa(4096)
                tree.evict_full(8192)
                tree.take_releases()
            else:
                tree.evict(4096, swa_only=True)
                tree.evict(8192)
                tree.releases()
            ops += 2
    return ops, toks


def run_radix(args, rank, world):
    """Host-side SWA radix prefix cache: native tree vs the oracle tree."""
    from hybrid_sliding_window_gb300 import api
    from oracle.radix import RadixSWA as OracleRadix
    n = max(64, 64 * args.steps)
    warm = radix_requests(16, 1)
    for _ in range(args.warmup):
        radix_ops(api.RadixSWA(64, 127), warm)
    reqs = radix_requests(n, 7)
    t0 = time.perf_counter()
    ops, toks = radix_ops(api.RadixSWA(64, 127), reqs)
    dt = time.perf_counter() - t0
    n_o = 16
    t1 = time.perf_counter()
    ops_o, _ = radix_ops(OracleRadix(64, 127), reqs[:n_o])
    dto = time.perf_counter() - t1
    return {
        "metric": "SWA radix prefix cache ops/s (match + insert + eviction)", "value": round(ops / dt, 1),
        "unit": "ops/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32 tokens / int64 slots",
        "data": "synthetic",
        "config": {"workload": f"{n} requests = one of 16 shared 2048-token prompts + 1024 own "
                               "tokens, page 64, window 127, SWA then full eviction every 8 "
                               "requests; host C++ tree in libswa (no device work)",
                   "tokens_per_s": round(toks / dt, 1)},
        "cpu_baseline": {"value": round(ops_o / dto, 1), "unit": "ops/s", "cores": 1,
                         "kind": "oracle", "sample": f"{n_o} requests of the same traffic"},
        "gpu_launches": 0,
    }


def translate_rate(st, n=1 << 24):
    """Kernel-facing id translation through a page table (one entry per page
    of the full pool, 10 % tombstones) for 16M random virtual ids: ids/s."""
    import torch
    from hybrid_sliding_window_gb300 import api
    g = torch.Generator(device=st.dev).manual_seed(5)
    pages = st.size_full // st.ps
    v2p = torch.randperm(pages, device=st.dev, generator=g) + 1
    v2p[torch.rand(pages, device=st.dev, generator=g) < 0.1] = -1
    virt = torch.randint(0, pages * st.ps, (n,), device=st.dev, generator=g)
    out = torch.empty_like(virt)
    mult = 2 * sum(1 for k, _, _ in st.spec.layers if k == 0)
    for _ in range(3):
        api.swa_translate_for_kernel(v2p, virt, st.ps, mult, out)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record()
    api.swa_translate_for_kernel(v2p, virt, st.ps, mult, out)
    a1.record()
    torch.cuda.synchronize()
    ms = a0.elapsed_time(a1)
    return {"ids": n, "ms": round(ms, 4), "ids_per_s": round(n / (ms / 1e3), 1),
            "bytes_per_id": 24}


def spec_alloc_rate(st):
    """One speculative decode step's allocation over the whole batch (a draft
    tree of 4 branches x 3 steps, 8 draft tokens: alloc_len slots per request
    through swa_alloc_extend), timed with CUDA events; the drafts' new pages
    are returned afterwards."""
    import numpy as np
    import torch
    from hybrid_sliding_window_gb300 import api
    ps = st.ps
    L = api.swa_decode_alloc_sizes(1, 3, 4, 8, True, ps)[0]
    pre = st.lens.copy()
    seq = pre + L
    if int(seq.max()) > st.rt.shape[1]:
        return None
    n = int(st.B * L)
    out_f = torch.empty(n, dtype=torch.int64, device=st.dev)
    out_s = torch.empty(n, dtype=torch.int64, device=st.dev)
    d_pre = torch.tensor(pre, device=st.dev)
    d_seq = torch.tensor(seq, device=st.dev)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a0.record()
    api.swa_alloc_extend(st.ctx, d_pre, d_seq, None, pre, seq, out_f, out_s,
                         req_to_token=st.rt, req_idx=st.rows_d)
    a1.record()
    torch.cuda.synchronize()
    ms = a0.elapsed_time(a1)
    # Return the drafts' whole new pages (positions from the next page boundary on).
    keep = -(-pre // ps) * ps
    idx = torch.cat([st.rt[int(r), int(k):int(s)].to(torch.int64)
                     for r, k, s in zip(st.rows, keep, seq)])
    pages = int((-(-(seq - keep) // ps)).sum())
    if idx.numel():
        api.swa_free(st.ctx, idx, pages, 0 if st.swa_ring else pages)
    for r, p in zip(st.rows, pre):
        st.rt[int(r), int(p):].zero_()
    assert api.swa_device_check(st.ctx) == 0
    return {"alloc_len": int(L), "slots": n, "ms": round(ms, 4),
            "slots_per_s": round(n / (ms / 1e3), 1)}


# Sources of the dominant kernel of each bench line: its DRAM traffic, taken
# from an ncu capture and stored under profiles/, is reported only while
# these files are unchanged since the capture.
DECODE_SOURCES = ("attn_decode_mma.cu", "split_merge.cuh", "kv_codec.cuh", "swa_internal.h")
EXTEND_SOURCES = ("attn_extend_tc.cu", "swa_internal.h")


def kernel_hash(files):
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "hybrid_sliding_window_gb300", "csrc")
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(name, files):
    """DRAM bytes (read + write) per launch from a stored ncu summary, or None
    when the kernel's sources changed since it was taken."""
    tp = os.path.join(ROOT, "profiles", name)
    try:
        with open(tp) as f:
            tj = json.load(f)
        if tj.get("kernel_source_hash") == kernel_hash(files):
            return tj["bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


# ------------------------------------------------------------- reference ---
def run_reference(args, rank, world):
    """The oracle on the host's cores: each step is the oracle's whole decode
    step of one request of the workload (eviction pass, alloc_decode, window
    translation, store encoding and attention on every layer), requests in a
    fixed seeded order; value = attended K+V bytes / oracle time."""
    if rank != 0:
        return None
    _pin_blas()
    import numpy as np
    from hybrid_sliding_window_gb300.workloads import SPECS
    spec = SPECS[args.workload]
    K, W = args.steps, args.warmup
    order = [int(i) for i in np.random.default_rng(7).permutation(spec.batch)]
    secs, nbytes = 0.0, 0
    for i in range(W + K):
        ph, nb, _ = oracle_request_step(args.workload, order[i % len(order)])
        if i >= W:
            secs += sum(ph.values())
            nbytes += nb
    v = nbytes / secs / 1e9
    model, ncpu = cpu_model()
    sample = (f"{K} whole per-request decode steps of the workload (plus {W} warm-up), "
              f"{nbytes / 1e9:.2f} GB of attended K+V in {secs:.1f} s of float64 numpy oracle "
              f"time on one core of {ncpu} ({model})")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(secs * 1e3 / K, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": spec.description},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="mimo",
                    choices=["mimo", "gptoss", "llama4", "tiny", "extend", "radix"])
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--separate-store", action="store_true",
                    help="decode steps call swa_store_kv and swa_attn_decode separately instead of "
                         "swa_store_kv_attn_decode")
    ap.add_argument("--no-extend", action="store_true",
                    help="skip the extend / evict figures added to the decode line")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the GPT-OSS, Llama4 and Tiny objects added to the MiMo line")
    ap.add_argument("--graph-steps", type=int, default=20,
                    help="decode steps captured in one CUDA graph and replayed once (0 = skip)")
    ap.add_argument("--steady-steps", type=int, default=160,
                    help="decode steps of the steady-state run that crosses the eviction "
                         "interval (0 = skip)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--batch", type=int, default=0, help="reduced batch (profiling only)")
    ap.add_argument("--layers", type=int, default=0, help="first N layers (profiling only)")
    ap.add_argument("--r", type=float, default=0.0, help="SWA/full token ratio (profiling only)")
    ap.add_argument("--chunk", type=int, default=0, help="prefill chunk (profiling only)")
    ap.add_argument("--swa-ring", action="store_true",
                    help="per-request SWA rings instead of the paged SWA pool")
    ap.add_argument("--attn-path", type=int, default=-1,
                    help="-1 best kernels (default); 1 cp.async decode; 0 generic (diagnostics)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "native":
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.workload == "extend":
        line = run_extend(args, rank, world)
    elif args.workload == "radix":
        line = run_radix(args, rank, world) if rank == 0 else None
    else:
        line = run_native(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "native":
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
