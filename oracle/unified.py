"""Oracle: the unified FULL/SWA pool allocated from both ends of one page range.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What the pages fix ([Pools 15], allocator-family table and the note on
``UnifiedSWAAllocatorBase``; [PR 34602], multi_ended_allocator.py):

* ``UnifiedSWATokenToKVPoolAllocator``: FULL and SWA share one id space and
  are allocated from the two ends;
* the shared virtual ids make the full->SWA mapping table disappear; the cost
  moves into the allocation policy, which has to manage both sub-pools'
  budgets at once;
* ``MultiEndedAllocator`` owns ``virtual_to_physical`` (one entry per virtual
  page); kernels address ``kernel_id(t) = v2p[t // ps] * (ps * multiplier) +
  t % ps`` with a tombstone page (-1) clamped to 0, the page-0 sink.

Readings where the pages stop (the plain ones; listed with the other
readings of the build):

* one physical page range ``1 .. P`` (page 0 is the sink of both sides).  The
  FULL side takes pages upward from the low end (its frontier ``low`` is the
  highest page it has taken, 0 at start), the SWA side downward from the high
  end (``high`` is the lowest page it has taken, P + 1 at start); the pages
  strictly between the two frontiers (``gap = high - low - 1``) belong to
  neither side;
* each side keeps the pages it released as a set and reuses the one nearest
  its own end first (FULL the lowest, SWA the highest: address-ordered first
  fit from each end), then takes from its frontier; after a release, a
  frontier that borders released pages of its own side retracts over them,
  returning them to the gap - so the two sides share the budget, and an
  allocation that needs ``n`` new pages on both sides fits iff
  ``max(0, n - |released_FULL|) + max(0, n - |released_SWA|) <= gap`` and
  ``n`` virtual pages are free;
* the FULL side owns the ids (the pages' ``is_id_owner``): virtual pages
  ``1 .. P`` come from a third free list, front first, released like the
  physical ones (distinct ids in ascending order, prepended);
* ``alloc_extend`` assigns virtual slots by the same statement as the
  two-pool allocator (a prefix ending inside a page continues after
  ``last_loc``; every other position opens the next new virtual page, pages
  in request order) and gives every new virtual page one FULL and one SWA
  physical page, in that order;
* ``free_swa`` releases the SWA page of each distinct virtual page of its
  slots that still has one and marks it a tombstone (-1); ``free`` does
  ``free_swa``, then releases each distinct virtual page's FULL page and the
  virtual page itself (FULL pages first, then the ids);
* out-of-window eviction is the two-pool rule (``allocator.evict_range``)
  over ``req_to_token`` holding virtual slots, each range released by
  ``free_swa``.
"""
from __future__ import annotations

from . import allocator as A

FULL = "full"
SWA = "swa"


class UnifiedNoMem(Exception):
    pass


class MultiEndedPool:
    def __init__(self, num_pages: int, page_size: int):
        self.P = int(num_pages)
        self.page_size = int(page_size)
        self.low = 0
        self.high = self.P + 1
        self.released = {FULL: [], SWA: []}
        self.vfree = list(range(1, self.P + 1))
        # virtual page -> physical page per side; -1 none / tombstone; the
        # sink virtual page 0 maps to the sink physical page 0.
        self.v2p = {FULL: [0] + [-1] * self.P, SWA: [0] + [-1] * self.P}

    # -- budget ------------------------------------------------------------------
    def gap(self) -> int:
        return self.high - self.low - 1

    def fits(self, n: int) -> bool:
        nf, ns = len(self.released[FULL]), len(self.released[SWA])
        return (n <= len(self.vfree)
                and max(0, n - nf) + max(0, n - ns) <= self.gap())

    def available_size(self) -> int:
        """Tokens of the largest whole-page allocation that fits on both sides."""
        n = 0
        while n < len(self.vfree) and self.fits(n + 1):
            n += 1
        return n * self.page_size

    # -- pages -----------------------------------------------------------------------
    def _take(self, side: str) -> int:
        if self.released[side]:      # kept ascending: nearest page to the side's end
            return self.released[side].pop(0 if side == FULL else -1)
        assert self.gap() > 0
        if side == FULL:
            self.low += 1
            return self.low
        self.high -= 1
        return self.high

    def _release(self, side: str, pages) -> None:
        pages = sorted(set(int(p) for p in pages))
        if not pages:
            return
        self.released[side] = sorted(self.released[side] + pages)
        if side == FULL:
            while self.low > 0 and self.low in self.released[FULL]:
                self.released[FULL].remove(self.low)
                self.low -= 1
        else:
            while self.high <= self.P and self.high in self.released[SWA]:
                self.released[SWA].remove(self.high)
                self.high += 1

    # -- allocation --------------------------------------------------------------------
    def alloc_extend(self, prefix_lens, seq_lens, last_loc):
        """Virtual slots of positions pre..seq-1 of each request, in request
        order; raises :class:`UnifiedNoMem` with nothing changed."""
        ps = self.page_size
        pre = [int(x) for x in prefix_lens]
        seq = [int(x) for x in seq_lens]
        last = [int(x) for x in last_loc]
        deltas = [A.ceil_div(s, ps) - A.ceil_div(p, ps) for p, s in zip(pre, seq)]
        total = sum(deltas)
        if not self.fits(total):
            raise UnifiedNoMem(total)
        vp = self.vfree[:total]
        self.vfree = self.vfree[total:]
        for v in vp:
            self.v2p[FULL][v] = self._take(FULL)
            self.v2p[SWA][v] = self._take(SWA)
        out, off = [], 0
        for r in range(len(pre)):
            out += A.extend_slots_plain(pre[r], seq[r], last[r], vp[off:off + deltas[r]], ps)
            off += deltas[r]
        return out

    def alloc_decode(self, seq_lens, last_loc):
        return self.alloc_extend([int(s) - 1 for s in seq_lens], seq_lens, last_loc)

    # -- release -----------------------------------------------------------------------
    def free_swa(self, virt) -> None:
        ps = self.page_size
        vs = sorted(set(int(t) // ps for t in virt))
        pages = []
        for v in vs:
            p = self.v2p[SWA][v]
            if v > 0 and p > 0:
                pages.append(p)
                self.v2p[SWA][v] = -1
        self._release(SWA, pages)

    def free(self, virt) -> None:
        ps = self.page_size
        self.free_swa(virt)
        vs = sorted(set(int(t) // ps for t in virt))
        pages, ids = [], []
        for v in vs:
            p = self.v2p[FULL][v]
            if v > 0 and p > 0:
                pages.append(p)
                ids.append(v)
                self.v2p[FULL][v] = -1
        self._release(FULL, pages)
        if ids:
            self.vfree = ids + self.vfree

    # -- lookups ---------------------------------------------------------------------------
    def physical_slot(self, side: str, t: int) -> int:
        """Slot of virtual token t in the side's own page units (-1 when the
        side holds no page for it)."""
        p = self.v2p[side][int(t) // self.page_size]
        return p * self.page_size + int(t) % self.page_size if p >= 0 else -1

    def check(self) -> None:
        """Conservation: every page of 1..P is owned by exactly one of FULL
        (live or in its free list, all at or below low), SWA (likewise, at or
        above high) or the gap; every virtual page is live or free once."""
        live_f = [p for p in self.v2p[FULL][1:] if p > 0]
        live_s = [p for p in self.v2p[SWA][1:] if p > 0]
        own_f = live_f + self.released[FULL]
        own_s = live_s + self.released[SWA]
        assert sorted(own_f) == list(range(1, self.low + 1)), "FULL pages"
        assert sorted(own_s) == list(range(self.high, self.P + 1)), "SWA pages"
        assert self.low < self.high
        live_v = [v for v in range(1, self.P + 1) if self.v2p[FULL][v] > 0]
        assert sorted(live_v + self.vfree) == list(range(1, self.P + 1)), "virtual pages"
        assert all(self.v2p[FULL][v] > 0 or self.v2p[SWA][v] <= 0 for v in range(1, self.P + 1))


def evict_swa(pool: MultiEndedPool, req_to_token, req_idx, pre_lens, evicted, protected,
              window_excl: int, interval: int, radix: bool = False):
    """The two-pool eviction pass over virtual slots: per request in batch
    order, ``free_swa(req_to_token[req, old:new])``, then ``evicted = new``."""
    out = [int(e) for e in evicted]
    for b in range(len(req_idx)):
        old, new = A.evict_range(int(pre_lens[b]), out[b], int(protected[b]), window_excl,
                                 pool.page_size, interval, radix)
        if new > old:
            row = req_to_token[int(req_idx[b])]
            pool.free_swa([int(row[t]) for t in range(old, new)])
            out[b] = new
    return out
