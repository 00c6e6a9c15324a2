"""Oracle: the two KV pools, the KV store and attention read through the
index tables.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

* Layout "per_layer" ([Pools 15], "second mapping: the KV store", MHA pool):
  one K and one V array per layer, each ``(size + page_size, H, D)``; slot 0
  (page 0) takes padded writes.
* Layout "envelope" ([PR 34602]): one byte buffer per pool of page
  envelopes, addressed through ``oracle.envelope.row_of``.

Full layers live in the full pool and are addressed by full slots; sliding
and chunked layers live in the SWA pool and are addressed by SWA slots, which
the caller translates once per batch ([SWA note], "attention backend:
translate once before reading or writing"; [Pools 15], "who writes into the
pages": the write target carries both locations).
"""
from __future__ import annotations

import numpy as np

from . import attention as A
from . import codecs as C
from . import envelope as E

STORE = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}
ITEM = {"f32": 4, "bf16": 2, "e4m3": 1}


class OraclePools:
    def __init__(self, layers, size_full: int, size_swa: int, page_size: int,
                 head_dim: int, dtype: str = "bf16", layout: str = "per_layer"):
        """``layers``: list of ``(kind, window, hkv)`` per model layer."""
        self.layers = list(layers)
        self.ps = page_size
        self.D = head_dim
        self.dtype = dtype
        self.layout = layout
        self.size = {True: size_full, False: size_swa}
        # Index of each layer inside its own pool.
        self.pool_layer = []
        counts = {True: 0, False: 0}
        for kind, _, _ in self.layers:
            is_full = kind == A.FULL
            self.pool_layer.append(counts[is_full])
            counts[is_full] += 1
        self.pool_layers = counts
        if layout == "per_layer":
            self.k = []
            self.v = []
            for kind, _, hkv in self.layers:
                n = self.size[kind == A.FULL] + page_size
                self.k.append(np.zeros((n, hkv, head_dim), STORE[dtype]))
                self.v.append(np.zeros((n, hkv, head_dim), STORE[dtype]))
        elif layout == "envelope":
            hkvs = {kind == A.FULL: hkv for kind, _, hkv in self.layers}
            for is_full in (True, False):
                for kind, _, hkv in self.layers:
                    if (kind == A.FULL) == is_full:
                        assert hkv == hkvs[is_full], "one head count per pool"
            self.hkv_pool = hkvs
            self.raw = {}
            for is_full in (True, False):
                L = counts[is_full]
                if L == 0:
                    continue
                row_bytes = hkvs[is_full] * head_dim * ITEM[dtype]
                pages = self.size[is_full] // page_size + 1
                nbytes = (E.envelope_bytes(pages, page_size, L, row_bytes)
                          + E.tail_pad_bytes(page_size, L, row_bytes))
                E.check_envelope(pages, page_size, L, head_dim, head_dim,
                                 row_bytes, nbytes)
                self.raw[is_full] = np.zeros(nbytes, np.uint8)
        else:
            raise ValueError(layout)

    # -- element codecs --------------------------------------------------------
    def encode(self, x, scale: float) -> np.ndarray:
        x = np.asarray(x, dtype=np.float32)
        if self.dtype == "f32":
            return x.copy()
        if self.dtype == "bf16":
            return C.bf16_encode(x)
        return C.e4m3_encode(x, scale)

    def decode(self, codes, scale: float) -> np.ndarray:
        if self.dtype == "f32":
            return np.asarray(codes, dtype=np.float64)
        if self.dtype == "bf16":
            return C.bf16_decode(codes).astype(np.float64)
        return C.e4m3_decode(codes) * float(scale)

    # -- row access --------------------------------------------------------------
    def _rows(self, layer: int, is_v: bool, slots):
        """Views onto the stored rows of ``slots`` (list of arrays)."""
        kind, _, hkv = self.layers[layer]
        if self.layout == "per_layer":
            buf = self.v[layer] if is_v else self.k[layer]
            return [buf[s] for s in slots]
        is_full = kind == A.FULL
        L = self.pool_layers[is_full]
        raw = self.raw[is_full]
        row_elems = hkv * self.D
        item = ITEM[self.dtype]
        out = []
        for s in slots:
            r = E.row_of(self.pool_layer[layer], is_v, int(s), self.ps, L)
            b0 = r * row_elems * item
            out.append(raw[b0:b0 + row_elems * item].view(STORE[self.dtype])
                       .reshape(hkv, self.D))
        return out

    def store(self, layer: int, k, v, full_loc, swa_loc, k_scale=1.0,
              v_scale=1.0) -> None:
        """Write rows ``k[i], v[i]`` ([n, Hkv, D]) of new token i at its
        location in this layer's pool."""
        kind = self.layers[layer][0]
        slots = full_loc if kind == A.FULL else swa_loc
        kc = self.encode(k, k_scale)
        vc = self.encode(v, v_scale)
        for i, s in enumerate(slots):
            self._rows(layer, False, [s])[0][...] = kc[i]
            self._rows(layer, True, [s])[0][...] = vc[i]

    def read(self, layer: int, slots, k_scale=1.0, v_scale=1.0):
        K = np.stack([self.decode(r, k_scale) for r in self._rows(layer, False, slots)])
        V = np.stack([self.decode(r, v_scale) for r in self._rows(layer, True, slots)])
        return K, V


def attention_through_tables(pools: OraclePools, alloc, layer: int,
                             req_to_token, req_idx, positions, q, sinks,
                             scale: float, k_scale=1.0, v_scale=1.0):
    """Attention of queries ``(b, p)`` (batch entry b at position p, q[i] of
    shape [Hq, D]) on ``layer``, reading keys through ``req_to_token`` and,
    on SWA-pool layers, the mapping.  Every in-window key must have a live SWA
    slot (evicted tokens map to 0): an assertion pins that eviction never
    frees what a later query reads."""
    kind, window, _ = pools.layers[layer]
    out = []
    for (b, p), qi in zip(positions, q):
        row = req_to_token[int(req_idx[b])]
        J = A.key_positions(kind, window, int(p))
        slots = [int(row[j]) for j in J]
        if kind != A.FULL:
            slots = [alloc.mapping[s] for s in slots]
            assert all(s > 0 for s in slots), "in-window key has no SWA slot"
        K, V = pools.read(layer, slots, k_scale, v_scale)
        out.append(A.attend_heads(np.asarray(qi, np.float64), K, V, sinks, scale))
    return np.stack(out)
