"""Oracle: page-major envelope addressing ([PR 34602], "implementation",
step 1 and the ``build_mha_views`` / ``translate_kv_loc_for_kernel``
excerpts).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

One pool is one byte buffer of page envelopes ``[L0_K*ps | L0_V*ps | L1_K*ps
| ...]``.  With equal K and V row widths the envelope is a uniform array of
``2L`` row-blocks per page, so every layer's K (block ``2l``) and V (block
``2l+1``) can be read as a dense ``(n_rows, H, D)`` view whose row for slot
``t`` is ``kernel_id(t) = (t // ps) * (ps * 2L) + t % ps``; the view of block
``b`` starts ``b * ps`` rows into the buffer.  The last view overshoots the
last page envelope by ``(2L - 1) * ps`` rows, so one page envelope of tail
pad follows the buffer.  Row ids must stay below ``2**31``; K and V widths
must match.
"""
from __future__ import annotations


class EnvelopeError(Exception):
    pass


def kernel_id(t: int, ps: int, num_layers: int) -> int:
    return (t // ps) * (ps * 2 * num_layers) + t % ps


def row_of(layer: int, is_v: bool, t: int, ps: int, num_layers: int) -> int:
    """Row (in ``H*D``-element units from the buffer start) holding slot t
    of ``layer``'s K or V: the dense view of block ``2l + is_v`` indexed at
    ``kernel_id(t)``."""
    block = 2 * layer + (1 if is_v else 0)
    return block * ps + kernel_id(t, ps, num_layers)


def row_of_strided(layer: int, is_v: bool, t: int, ps: int,
                   num_layers: int) -> int:
    """The same row through an independent 4-D strided index
    ``[page][block][t % ps]`` (the pages' test compares the dense views with
    such a strided reference)."""
    page = t // ps
    block = 2 * layer + (1 if is_v else 0)
    blocks = 2 * num_layers
    return (page * blocks + block) * ps + (t % ps)


def envelope_bytes(num_pages_total: int, ps: int, num_layers: int,
                   row_bytes: int) -> int:
    """Bytes of the buffer proper (``num_pages_total`` envelopes)."""
    return num_pages_total * 2 * num_layers * ps * row_bytes


def tail_pad_bytes(ps: int, num_layers: int, row_bytes: int) -> int:
    """One page envelope: ``ps * entry_bytes`` with ``entry_bytes = 2L`` rows."""
    return ps * 2 * num_layers * row_bytes


def check_envelope(num_pages_total: int, ps: int, num_layers: int,
                   head_dim: int, v_head_dim: int, row_bytes: int,
                   buffer_bytes: int) -> int:
    """Start-up checks; returns ``n_rows``."""
    if head_dim != v_head_dim:
        raise EnvelopeError("envelope views need head_dim == v_head_dim")
    n_rows = num_pages_total * 2 * num_layers * ps
    if n_rows >= 2 ** 31:
        raise EnvelopeError("kernel-facing row ids overflow int32")
    last_view_end = ((2 * num_layers - 1) * ps + n_rows) * row_bytes
    if last_view_end > buffer_bytes:
        raise EnvelopeError("buffer lacks the one-envelope tail pad")
    return n_rows


def translate_for_kernel(v2p, virt_tokens, ps: int, multiplier: int):
    """Kernel-facing ids of virtual token ids through a virtual-to-physical
    page table ([PR 34602], multi_ended_allocator.py,
    "translate_kv_loc_for_kernel"): id = phys * (ps * multiplier) + t % ps
    with phys = v2p[t // ps]; a tombstone page (phys = -1) clamps to 0, the
    page-0 sink.  ``multiplier`` is the row blocks of a page (2L)."""
    out = []
    for t in virt_tokens:
        t = int(t)
        phys = int(v2p[t // ps])
        out.append(max(0, phys * ps * multiplier + t % ps))
    return out
