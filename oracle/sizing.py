"""Oracle: two-pool sizing ([SWA note], "how memory is split:
--swa-full-tokens-ratio").

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

``r`` is a per-layer token-count ratio (SWA capacity / full capacity), not a
memory ratio.  With F and S the KV bytes of one token in one full / SWA layer
(``kv_heads * (head_dim + v_head_dim) * dtype_size``)::

    cell   = F * L_full + r * S * L_swa
    N_full = floor(M / cell)
    N_swa  = r * N_full

both aligned down to a page; an SWA pool with ``N_swa <= W + P`` cannot hold
one request and is a start-up error.
"""
from __future__ import annotations

import math


class SizingError(Exception):
    pass


def bytes_per_token_layer(kv_heads: int, head_dim: int, v_head_dim: int,
                          dtype_size: int) -> int:
    return kv_heads * (head_dim + v_head_dim) * dtype_size


def cell_bytes(F: float, S: float, L_full: int, L_swa: int, r: float) -> float:
    return F * L_full + r * S * L_swa


def pool_sizes(mem_bytes: int, F: int, S: int, L_full: int, L_swa: int,
               r: float, page_size: int, window: int):
    """Returns ``(N_full, N_swa)`` in tokens."""
    cell = cell_bytes(F, S, L_full, L_swa, r)
    n_full = math.floor(mem_bytes / cell)
    n_swa = math.floor(r * n_full)
    n_full = (n_full // page_size) * page_size
    n_swa = (n_swa // page_size) * page_size
    if n_swa <= window + page_size:
        raise SizingError(f"SWA pool of {n_swa} tokens holds no request "
                          f"(window {window}, page {page_size})")
    return n_full, n_swa
