"""Oracle: windowed / chunked-local / full attention with a sink, by brute force.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[SWA note], opening paragraph and "design": each query sees only the most
recent keys on a sliding layer; a full layer sees every earlier key; Llama4's
local layers attend within fixed chunks.  The engine's window length excludes
the current token ("model configs return sliding_window - 1"), so a sliding
layer with exclusive length ``Wx`` gives the query at position ``p`` the keys
``max(0, p - Wx) .. p``.  [SWA note], "design": a learnable per-head sink lets
a query leak weight out of the window; it enters the softmax denominator only.

For query head ``h`` (KV head ``h // G``, G = Hq / Hkv), score scale ``c``,
sink logit ``sigma_h`` and key set ``J``::

    s_j = c * <q_h, k_j>
    m   = max(max_j s_j, sigma_h)          (sigma_h omitted without a sink)
    o_h = sum_j exp(s_j - m) v_j / (exp(sigma_h - m) + sum_j exp(s_j - m))

All arithmetic is float64.
"""
from __future__ import annotations

import numpy as np

FULL = 0
SLIDING = 1
CHUNKED = 2


def key_positions(kind: int, window: int, p: int) -> range:
    """Positions a query at ``p`` attends.

    * FULL: ``0 .. p`` (causal).
    * SLIDING: ``max(0, p - window) .. p`` with ``window`` the exclusive
      length (keys before the current one).
    * CHUNKED: ``floor(p / C) * C .. p`` with ``window = C`` the chunk size
      (reading of the chunked-local mask: chunk-aligned blocks).
    """
    if kind == FULL:
        return range(0, p + 1)
    if kind == SLIDING:
        return range(max(0, p - window), p + 1)
    if kind == CHUNKED:
        return range((p // window) * window, p + 1)
    raise ValueError(kind)


def lookback(kind: int, window: int) -> int:
    """Largest ``p - j`` any query of this layer kind may need (the exclusive
    window used by eviction).  A chunked layer of chunk C needs at most C-1."""
    if kind == SLIDING:
        return window
    if kind == CHUNKED:
        return window - 1
    raise ValueError(kind)


def softmax_with_sink(scores: np.ndarray, sink) -> np.ndarray:
    """Weights of the keys (the sink's own weight is dropped)."""
    scores = np.asarray(scores, dtype=np.float64)
    m = scores.max() if scores.size else -np.inf
    if sink is not None:
        m = max(m, float(sink))
    e = np.exp(scores - m)
    denom = e.sum() + (np.exp(float(sink) - m) if sink is not None else 0.0)
    return e / denom


def attend_one(q: np.ndarray, K: np.ndarray, V: np.ndarray, sink, scale: float):
    """One query head against explicit key/value rows ``K[n, D]``, ``V[n, D]``."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    s = scale * (K @ q)
    w = softmax_with_sink(s, sink)
    return w @ V


def attend_heads(q: np.ndarray, K: np.ndarray, V: np.ndarray, sinks, scale: float):
    """All query heads of one query: ``q[Hq, D]``, ``K, V[n, Hkv, D]``.
    Query head ``h`` reads KV head ``h // (Hq // Hkv)``."""
    hq = q.shape[0]
    hkv = K.shape[1]
    assert hq % hkv == 0
    g = hq // hkv
    out = np.zeros((hq, q.shape[1]), dtype=np.float64)
    for h in range(hq):
        kv = h // g
        sink = None if sinks is None else float(sinks[h])
        out[h] = attend_one(q[h], K[:, kv, :], V[:, kv, :], sink, scale)
    return out
