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


# ---------------------------------------------------------------------------
# Per-step decode allocation under speculative decoding ("SGLang source
# teardown (15)", section "how the sizes are set: from the memory budget to
# pool sizes"): how many KV slots one request may take in one decode step,
# the per-step reserve, and the req_to_token row headroom.
SPEC_NONE, SPEC_DRAFT, SPEC_UNO = 0, 1, 2


def decode_alloc_len(algo: int, steps: int, topk: int, draft_tokens: int, page_size: int,
                     has_draft_kv: bool = True) -> int:
    """Slots one request allocates per decode step.

    * no speculation: one token;
    * UNO: its draft tokens plus one extra clean-root position;
    * page size 1, a single branch, or drafts without KV of their own: the
      larger of steps x topk and the draft-token count;
    * otherwise (pages of more than one slot and several branches): every
      branch may start anywhere inside a page, so it can touch
      ceil((page_size - 1 + steps) / page_size) pages, and each branch gets
      its own pages: that many pages x page_size x topk, or the draft-token
      count if larger.
    """
    if algo == SPEC_NONE:
        return 1
    steps = max(int(steps), 1)
    topk = max(int(topk), 1)
    if algo == SPEC_UNO:
        if draft_tokens is None:
            raise ValueError("UNO needs the draft-token count")
        return int(draft_tokens) + 1
    d = int(draft_tokens or 0)
    if page_size == 1 or topk == 1 or not has_draft_kv:
        return max(steps * topk, d)
    pages_per_branch = -(-(page_size - 1 + steps) // page_size)
    return max(pages_per_branch * page_size * topk, d)


def decode_reserve(algo, steps, topk, draft_tokens, page_size, has_draft_kv=True) -> int:
    """Reserve per request per step: twice the allocation (a double buffer for
    the scheduler's committed length lagging the device under overlap)."""
    return 2 * decode_alloc_len(algo, steps, topk, draft_tokens, page_size, has_draft_kv)


def req_to_token_extra(algo, steps, topk, draft_tokens, page_size, has_draft_kv=True) -> int:
    """Columns of headroom a req_to_token row needs past the context length:
    4 + the draft-token count, raised for speculation on pages larger than one
    slot (or UNO) to the per-step reserve plus page_size - 1 (the allocation
    may be rounded up to a page)."""
    d = int(draft_tokens or 0)
    extra = 4 + d
    if algo != SPEC_NONE and (page_size > 1 or algo == SPEC_UNO):
        extra = max(extra, decode_reserve(algo, steps, topk, draft_tokens, page_size,
                                          has_draft_kv) + page_size - 1)
    return extra
