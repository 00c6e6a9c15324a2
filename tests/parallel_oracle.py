"""Oracle attention for many queries at once, spread over the host's cores.

Test infrastructure: each job is one (layer, request, KV head) with one or
more query positions; a worker redraws that head's K and V at the attended
positions from the seeded generator (``synth``) and runs the oracle's
brute-force softmax (``oracle.attention.attend_one``) for every query head of
the group.  Workers are started with ``spawn`` (the parent has a CUDA
context).  Nothing here reads the GPU.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _draw(job, stream, J):
    from hybrid_sliding_window_gb300 import synth
    from oracle import codecs as OC
    x = synth.tokens_head(job["seed"], stream, job["layer"], job["row"], J, job["kvh"],
                          job["D"], bf16=job["dtype"] != "f32").astype(np.float64)
    if job["dtype"] == "e4m3":
        x = OC.e4m3_decode(OC.e4m3_encode(x.astype(np.float32))).astype(np.float64)
    return x


def _run(job):
    from hybrid_sliding_window_gb300 import synth
    from oracle import attention as OT
    ranges = [OT.key_positions(job["kind"], job["window"], int(p)) for p in job["pos"]]
    lo = min(r.start for r in ranges)
    hi = max(r.stop for r in ranges)
    J = np.arange(lo, hi, dtype=np.int64)
    K = _draw(job, synth.STREAM_K, J)
    V = _draw(job, synth.STREAM_V, J)
    q = np.asarray(job["q"], np.float64)            # [nq, G, D]
    sinks = job["sinks"]
    out = np.empty(q.shape, np.float64)
    for i, r in enumerate(ranges):
        Ks, Vs = K[r.start - lo:r.stop - lo], V[r.start - lo:r.stop - lo]
        for g in range(q.shape[1]):
            out[i, g] = OT.attend_one(q[i, g], Ks, Vs,
                                      None if sinks is None else float(sinks[g]), job["scale"])
    return out


def attend_jobs(jobs, procs=None):
    """Oracle outputs ``[nq, G, D]`` (float64) for each job, in order."""
    if not jobs:
        return []
    n = procs or min(len(jobs), os.cpu_count() or 1, 32)
    if n <= 1:
        return [_run(j) for j in jobs]
    # One BLAS thread per worker (the variables are read when a worker
    # imports numpy, so they are set before the workers start).
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: "1" for k in keys})
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            return pool.map(_run, jobs, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def decode_jobs(spec, layer, rows, seq_h, q_cpu, sinks_h, scale):
    """One job per (request, KV head) of a decode step at positions seq - 1.
    q_cpu: [B, Hq, D] query values drawn on the CPU."""
    kind, w, hkv = spec.layers[layer]
    G = spec.Hq // hkv
    okind = {0: 0, 1: 1, 2: 2}[int(kind)]
    jobs = []
    for b, row in enumerate(rows):
        for h in range(hkv):
            jobs.append(dict(seed=spec.seed, layer=layer, row=int(row), kvh=h, D=spec.D,
                             dtype=spec.dtype, kind=okind, window=int(w),
                             pos=[int(seq_h[b]) - 1], q=q_cpu[b:b + 1, h * G:(h + 1) * G],
                             sinks=None if sinks_h is None else sinks_h[h * G:(h + 1) * G],
                             scale=scale, b=b, h=h))
    return jobs
