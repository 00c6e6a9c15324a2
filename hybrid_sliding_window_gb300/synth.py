"""Seeded synthetic inputs (numpy side).

This module holds no arithmetic of the attention / allocation method: it only
draws the q, k, v and sink values the workloads feed in.  A GPU kernel
(``swa_synth_tokens`` in the C library) implements the same generator, so
large inputs can be drawn on the device and any sampled element redrawn here.

Generator (counter based, no state):

* ``mix64`` is the SplitMix64 output function (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014).
* ``base = mix64((seed << 32) ^ stream)``;  element ``i`` draws
  ``z = mix64(base + (i + 1) * 0x9E3779B97F4A7C15)`` (mod 2**64).
* The four 16-bit fields of ``z`` are summed (Irwin-Hall, n = 4) and mapped to
  an approximately standard normal value in float32:
  ``(sum - 131070) * float32(sqrt(3) / 65536)``; both factors are exact in
  float32, so the single correctly rounded product is identical on any IEEE
  machine.  bf16 inputs are that value rounded to nearest even.
* Element index of token ``(layer, req, pos, head, dim)``:
  ``layer << 47 | req << 35 | pos << 15 | head << 8 | dim``
  (layer < 128, req < 4096, pos < 2**20, head < 128, dim < 256).
"""
from __future__ import annotations

import numpy as np

STREAM_Q = 1
STREAM_K = 2
STREAM_V = 3
STREAM_SINK = 4

_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
NORMAL_SCALE = np.float32(np.sqrt(3.0) / 65536.0)


def mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def element_index(layer, req, pos, head, dim) -> np.ndarray:
    l = np.asarray(layer, dtype=np.uint64)
    r = np.asarray(req, dtype=np.uint64)
    p = np.asarray(pos, dtype=np.uint64)
    h = np.asarray(head, dtype=np.uint64)
    d = np.asarray(dim, dtype=np.uint64)
    return ((l << np.uint64(47)) | (r << np.uint64(35)) | (p << np.uint64(15))
            | (h << np.uint64(8)) | d)


def normal_f32(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    base = mix64(np.array([(int(seed) << 32) ^ int(stream)], dtype=np.uint64))[0]
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = mix64(base + (idx + np.uint64(1)) * _GAMMA)
    s = ((z & np.uint64(0xFFFF)) + ((z >> np.uint64(16)) & np.uint64(0xFFFF))
         + ((z >> np.uint64(32)) & np.uint64(0xFFFF)) + (z >> np.uint64(48)))
    centred = (s.astype(np.int64) - 131070).astype(np.float32)
    return (centred * NORMAL_SCALE).astype(np.float32)


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even), returned as float32."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)).astype(np.uint32)
    return r.view(np.float32)


def tokens(seed: int, stream: int, layer: int, reqs, positions, heads: int,
           dim: int, bf16: bool = True) -> np.ndarray:
    """Values ``[n, heads, dim]`` for tokens ``(reqs[i], positions[i])``."""
    reqs = np.asarray(reqs, dtype=np.int64).reshape(-1, 1, 1)
    pos = np.asarray(positions, dtype=np.int64).reshape(-1, 1, 1)
    h = np.arange(heads, dtype=np.int64).reshape(1, -1, 1)
    d = np.arange(dim, dtype=np.int64).reshape(1, 1, -1)
    idx = element_index(layer, reqs, pos, h, d)
    x = normal_f32(seed, stream, idx)
    return to_bf16_values(x) if bf16 else x


def tokens_head(seed: int, stream: int, layer: int, req: int, positions, head: int,
                dim: int, bf16: bool = True) -> np.ndarray:
    """Values ``[n, dim]`` of one head for tokens ``(req, positions[i])``:
    the ``head`` slice of ``tokens`` without drawing the other heads."""
    pos = np.asarray(positions, dtype=np.int64).reshape(-1, 1)
    d = np.arange(dim, dtype=np.int64).reshape(1, -1)
    x = normal_f32(seed, stream, element_index(layer, req, pos, head, d))
    return to_bf16_values(x) if bf16 else x


def sinks(seed: int, layer: int, num_q_heads: int) -> np.ndarray:
    """Per-head sink logits ``[Hq]`` of one layer (float32)."""
    return tokens(seed, STREAM_SINK, layer, [0], [0], num_q_heads, 1,
                  bf16=False).reshape(num_q_heads)


def permutation(seed: int, n: int, start: int = 1) -> np.ndarray:
    """A seeded permutation of ``start .. start + n - 1`` (int64), used to
    assign pool pages in a shuffled order."""
    rng = np.random.default_rng(seed)
    return (rng.permutation(n) + start).astype(np.int64)


def seq_lens_uniform(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def seq_lens_log_uniform(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))).astype(np.int64)
