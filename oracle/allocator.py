"""Oracle: free-page ledgers, the full->SWA mapping and the two-pool allocator.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Everything here is plain Python over lists / small numpy arrays, in the order
the pages describe it:

* one ledger per pool ([Pools 15], "third mapping: the page allocator"):
  pages ``1..num_pages`` (page 0 is the padding sink), allocation takes from
  the front, release either prepends the unique page ids in ascending order
  (what ``torch.unique`` returns) or, with ``need_sort``, stages them until a
  request finds the front list short, when the union is sorted
  ([Pools 15], "_release_page_ids: the switch for sort-merge");
  ``available_size = (free + staged) * page_size``.
* the mapping ([SWA note], "two pools and the mapping"; [Pools 15], "two pools
  plus mapping table"): ``size_full + page_size`` zeros followed by one ``-1``;
  0 means "no SWA slot"; looking up ``-1`` (no prefix) yields ``-1``.
* ``alloc`` / ``alloc_extend`` / ``alloc_decode`` allocate the same number of
  slots in both ledgers, the SWA side continuing from the translated
  ``last_loc``, then write ``mapping[full] = swa`` ([SWA note], same section).
* ``free`` releases full pages then calls ``free_swa``; ``free_swa`` releases
  only SWA slots whose mapping is > 0 and then zeroes the mapping, so
  ``free_swa`` followed by ``free`` never frees twice ([SWA note]).
* ``available_size`` is the minimum of the two pools ([SWA note]).
* out-of-window eviction ([SWA note], "runtime: returning slid-out KV").
"""
from __future__ import annotations

import numpy as np


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class OracleNoMem(Exception):
    """The pages' ``None`` return: not enough pages, nothing allocated."""


class PageLedger:
    """Free-page list of one pool ([Pools 15], PagedTokenToKVPoolAllocator).

    ``size`` is the token capacity; ``num_pages = size // page_size``.  With
    ``page_size == 1`` this is the token allocator of the same page (slots are
    pages).  ``initial`` replaces the default ``1..num_pages`` order (used to
    seed a permuted pool); it must be a permutation of ``1..num_pages``.
    """

    def __init__(self, size: int, page_size: int, need_sort: bool = False,
                 initial=None):
        self.page_size = int(page_size)
        self.num_pages = int(size) // self.page_size
        if initial is None:
            self.free = list(range(1, self.num_pages + 1))
        else:
            self.free = [int(x) for x in initial]
            assert sorted(self.free) == list(range(1, self.num_pages + 1))
        self.staged: list[list[int]] = []
        self.need_sort = bool(need_sort)

    # -- capacity --------------------------------------------------------
    def num_staged(self) -> int:
        return sum(len(s) for s in self.staged)

    def available_size(self) -> int:
        return (len(self.free) + self.num_staged()) * self.page_size

    # -- the sort-merge of staged pages ------------------------------------
    def merge_and_sort(self) -> None:
        if not self.staged:
            return
        union = list(self.free)
        for s in self.staged:
            union.extend(s)
        self.free = sorted(union)
        self.staged = []

    def ensure(self, n_pages: int) -> bool:
        """Merge staged pages when the front list is short (need_sort only),
        then report whether ``n_pages`` can be taken."""
        if self.need_sort and n_pages > len(self.free):
            self.merge_and_sort()
        return n_pages <= len(self.free)

    def take(self, n_pages: int) -> list[int]:
        assert n_pages <= len(self.free)
        out = self.free[:n_pages]
        self.free = self.free[n_pages:]
        return out

    # -- release ------------------------------------------------------------
    def release_pages(self, pages) -> None:
        pages = [int(p) for p in pages]
        if not pages:
            return
        if self.need_sort:
            self.staged.append(pages)
        else:
            self.free = pages + self.free

    def free_slots(self, slots) -> None:
        """``free(free_index)``: release ``unique(free_index // page_size)``."""
        slots = [int(s) for s in slots]
        if not slots:
            return
        pages = sorted(set(s // self.page_size for s in slots))
        self.release_pages(pages)

    def all_free_pages(self) -> list[int]:
        out = list(self.free)
        for s in self.staged:
            out.extend(s)
        return out


def extend_slots_plain(pre: int, seq: int, last_loc: int, new_pages: list[int],
                       ps: int) -> list[int]:
    """Slots of positions ``pre .. seq-1`` of one request, stated plainly.

    A position inside the page that is already open (the prefix does not end
    on a page boundary) continues right after ``last_loc``; every other
    position ``t`` lives in the ``(t // ps - ceil(pre / ps))``-th new page at
    offset ``t % ps`` (slot(p, k) = p * ps + k, [Pools 15], "alloc_extend").
    """
    open_end = ceil_div(pre, ps) * ps
    out = []
    for t in range(pre, seq):
        if t < open_end:
            out.append(last_loc + 1 + (t - pre))
        else:
            k = t // ps - ceil_div(pre, ps)
            out.append(new_pages[k] * ps + t % ps)
    return out


def extend_slots_three_part(pre: int, seq: int, last_loc: int,
                            new_pages: list[int], ps: int) -> list[int]:
    """The same slots built the way the pages' kernel builds them, in three
    parts ([Pools 15], "alloc_extend", Part 1/2/3): fill the half-full page
    from ``last_loc + 1``; write whole new pages; write the tail page, which
    is the last new page.  Kept separate so the two statements can be
    compared."""
    out = []
    n1 = min(seq, ceil_div(pre, ps) * ps) - pre
    for k in range(n1):
        out.append(last_loc + 1 + k)
    if pre + n1 == seq:
        return out
    n2 = (seq // ps) * ps - ceil_div(pre, ps) * ps
    for off in range(n2):
        out.append(new_pages[off // ps] * ps + off % ps)
    n3 = seq - (seq // ps) * ps
    if n3 > 0:
        tail_page = new_pages[len(new_pages) - 1]
        for k in range(n3):
            out.append(tail_page * ps + k)
    return out


class TwoPoolAllocator:
    """Full pool + SWA pool + full->SWA mapping ([SWA note]; [Pools 15],
    SWATokenToKVPoolAllocator)."""

    def __init__(self, size_full: int, size_swa: int, page_size: int,
                 need_sort: bool = False, init_full=None, init_swa=None):
        self.page_size = int(page_size)
        self.size_full = int(size_full)
        self.size_swa = int(size_swa)
        self.full = PageLedger(size_full, page_size, need_sort, init_full)
        self.swa = PageLedger(size_swa, page_size, need_sort, init_swa)
        # size + page_size zeros, then the trailing -1 sentinel.
        self.mapping = [0] * (self.size_full + self.page_size) + [-1]

    # -- lookups -------------------------------------------------------------
    def translate(self, full_idx):
        """``full_to_swa_index_mapping[idx]`` with Python indexing, so -1 reads
        the trailing sentinel."""
        if np.ndim(full_idx) == 0:
            return self.mapping[int(full_idx)]
        return [self.mapping[int(i)] for i in full_idx]

    def available_size(self) -> int:
        return min(self.full.available_size(), self.swa.available_size())

    # -- allocation ------------------------------------------------------------
    def _reserve(self, n_pages: int) -> None:
        ok_full = self.full.ensure(n_pages)
        ok_swa = self.swa.ensure(n_pages)
        if not (ok_full and ok_swa):
            raise OracleNoMem(n_pages)

    def alloc(self, need_size: int) -> list[int]:
        """Plain ``alloc(need_size)``: whole pages from both ledgers."""
        ps = self.page_size
        assert need_size % ps == 0
        n = need_size // ps
        self._reserve(n)
        fp = self.full.take(n)
        sp = self.swa.take(n)
        full_out = [p * ps + k for p in fp for k in range(ps)]
        swa_out = [p * ps + k for p in sp for k in range(ps)]
        for f, s in zip(full_out, swa_out):
            self.mapping[f] = s
        return full_out

    def alloc_extend(self, prefix_lens, seq_lens, last_loc, three_part=False):
        """Returns ``(full_slots, swa_slots)`` in request order, or raises
        :class:`OracleNoMem` leaving every ledger as it was (except for a
        need_sort merge, which the pages also perform before the check)."""
        ps = self.page_size
        pre = [int(x) for x in prefix_lens]
        seq = [int(x) for x in seq_lens]
        last = [int(x) for x in last_loc]
        assert len(pre) == len(seq) == len(last)
        deltas = [ceil_div(s, ps) - ceil_div(p, ps) for p, s in zip(pre, seq)]
        total = sum(deltas)
        self._reserve(total)
        fp = self.full.take(total)
        sp = self.swa.take(total)
        build = extend_slots_three_part if three_part else extend_slots_plain
        full_out, swa_out = [], []
        off = 0
        for r in range(len(pre)):
            nf = fp[off:off + deltas[r]]
            ns = sp[off:off + deltas[r]]
            off += deltas[r]
            swa_last = self.translate(last[r])
            full_out += build(pre[r], seq[r], last[r], nf, ps)
            swa_out += build(pre[r], seq[r], swa_last, ns, ps)
        for f, s in zip(full_out, swa_out):
            self.mapping[f] = s
        return full_out, swa_out

    def alloc_decode(self, seq_lens, last_loc):
        """One token per request: ``pre = seq - 1`` ([Pools 15],
        "alloc_decode")."""
        seq = [int(x) for x in seq_lens]
        return self.alloc_extend([s - 1 for s in seq], seq, last_loc)

    # -- release -----------------------------------------------------------------
    def free_swa(self, full_idx) -> None:
        idx = [int(i) for i in full_idx]
        if not idx:
            return
        swa = [self.mapping[i] for i in idx]
        self.swa.free_slots([s for s in swa if s > 0])
        for i in idx:
            self.mapping[i] = 0

    def free(self, full_idx) -> None:
        idx = [int(i) for i in full_idx]
        if not idx:
            return
        self.full.free_slots(idx)
        self.free_swa(idx)

    # -- debug invariant ([Pools 15], "free_group": no page twice) ---------------
    def check_no_duplicate_pages(self) -> None:
        for led in (self.full, self.swa):
            pages = led.all_free_pages()
            assert len(pages) == len(set(pages)), "duplicate free page"
            assert all(1 <= p <= led.num_pages for p in pages)


def evict_range(pre_len: int, evicted: int, protected: int, window_excl: int,
                page_size: int, interval: int, radix: bool = False):
    """Out-of-window range of one request ([SWA note], "runtime: returning
    slid-out KV").

    ``pre_len`` tokens already hold KV; the next query sits at ``pre_len``
    and needs keys from ``pre_len - window_excl`` on.  The upper bound is
    ``pre_len - window_excl`` (chunk cache) or ``pre_len - max(window_excl,
    page_size)`` (radix cache), aligned down to a page; the lower bound is
    ``max(evicted, protected)`` aligned up to a page, so a page holding
    protected tokens is never freed.  In decode (``interval > 0``) the pass
    only runs once at least ``interval`` tokens have slid out past
    ``evicted``; ``interval == 0`` means "always" (before a prefill chunk).

    Returns ``(old, new)``; nothing is freed unless ``new > old``.
    """
    ps = page_size
    bound = pre_len - (max(window_excl, ps) if radix else window_excl)
    if interval > 0 and bound - evicted < interval:
        return evicted, evicted
    new = (bound // ps) * ps if bound > 0 else 0
    old = ceil_div(max(evicted, protected), ps) * ps
    return old, new


def evict_swa(alloc: TwoPoolAllocator, req_to_token, req_idx, pre_lens,
              evicted, protected, window_excl: int, interval: int,
              radix: bool = False):
    """Run the eviction pass over a batch, request by request in batch
    order: ``free_swa(req_to_token[req, old:new])`` then advance ``evicted``.
    Returns the new ``evicted`` list and the number of SWA pages freed."""
    out = list(int(e) for e in evicted)
    freed = 0
    for b in range(len(req_idx)):
        old, new = evict_range(int(pre_lens[b]), out[b], int(protected[b]),
                               window_excl, alloc.page_size, interval, radix)
        if new > old:
            row = req_to_token[int(req_idx[b])]
            idx = [int(row[t]) for t in range(old, new)]
            before = alloc.swa.available_size()
            alloc.free_swa(idx)
            freed += (alloc.swa.available_size() - before) // alloc.page_size
            out[b] = new
    return out, freed


# ---------------------------------------------------------------------------
# Per-request SWA ring ("SGLang source teardown (15)", section "why sliding
# windows can be accounted per request": the SWA pool becomes one ring per
# request slot).
#
# The pages give the capacity rule: a ring costs ``ceil(ring_size / ps) * ps``
# slots and the SWA pool holds one ring per request slot.  They do not print
# the address of a position inside its ring; the reading taken here is the
# plain one: request slot ``r`` owns slots ``ps + r * cost .. ps + (r+1) *
# cost - 1`` (slot range 0..ps-1 stays the padding page, so mapping 0 still
# means "no SWA slot") and position ``t`` of that request lives at
# ``ps + r * cost + t % cost``.  Nothing is allocated or released on the SWA
# side; the mapping is still written (full slot -> ring slot) so translation,
# the per-batch plan and attention are unchanged, and eviction / free_swa
# only zero mapping entries.  Reading: a ring must hold the window plus every
# position stored before the attention that reads it, so a request may add at
# most ``cost - window_excl`` tokens per call.

def ring_cost(ring_size: int, page_size: int) -> int:
    """Slots one request's ring occupies: ring_size rounded up to a page."""
    return ceil_div(int(ring_size), int(page_size)) * int(page_size)


def ring_pool_size(req_slots: int, ring_size: int, page_size: int) -> int:
    """SWA pool capacity in ring mode: one ring per request slot."""
    return int(req_slots) * ring_cost(ring_size, page_size)


def ring_slot(req: int, pos: int, ring_size: int, page_size: int) -> int:
    """SWA slot of position ``pos`` of the request in slot ``req``."""
    cost = ring_cost(ring_size, page_size)
    return int(page_size) + int(req) * cost + int(pos) % cost


class _RingSide:
    """Stands where the SWA page ledger stands in paged mode: nothing to take
    or give back, the whole pool is always 'available'."""

    def __init__(self, size: int, page_size: int):
        self.page_size = int(page_size)
        self.size = int(size)
        self.num_pages = self.size // self.page_size

    def available_size(self) -> int:
        return self.size

    def free_slots(self, slots) -> None:
        pass

    def all_free_pages(self) -> list[int]:
        return []


class RingTwoPoolAllocator(TwoPoolAllocator):
    """Full pool (paged, as in :class:`TwoPoolAllocator`) + per-request SWA
    rings.  ``window_excl`` is the largest lookback of the SWA-pool layers;
    ``ring_size`` must be at least ``window_excl + 1``."""

    def __init__(self, size_full: int, page_size: int, ring_size: int, req_slots: int,
                 window_excl: int, need_sort: bool = False, init_full=None):
        if ring_size < window_excl + 1:
            raise ValueError("ring smaller than the window")
        self.ring_size = int(ring_size)
        self.req_slots = int(req_slots)
        self.window_excl = int(window_excl)
        self.cost = ring_cost(ring_size, page_size)
        super().__init__(size_full, ring_pool_size(req_slots, ring_size, page_size), page_size,
                         need_sort, init_full, None)
        self.swa = _RingSide(self.size_swa, page_size)

    def available_size(self) -> int:
        return self.full.available_size()

    def alloc(self, need_size: int):
        raise ValueError("plain alloc has no request slot in ring mode")

    def alloc_extend(self, prefix_lens, seq_lens, last_loc, req_idx=None, three_part=False):
        ps = self.page_size
        pre = [int(x) for x in prefix_lens]
        seq = [int(x) for x in seq_lens]
        last = [int(x) for x in last_loc]
        reqs = [int(x) for x in req_idx]
        assert len(pre) == len(seq) == len(last) == len(reqs)
        for p, s, r in zip(pre, seq, reqs):
            if not 0 <= r < self.req_slots:
                raise ValueError("request slot outside the rings")
            if s - p + self.window_excl > self.cost:
                raise ValueError("more new tokens than the ring holds beside the window")
        deltas = [ceil_div(s, ps) - ceil_div(p, ps) for p, s in zip(pre, seq)]
        total = sum(deltas)
        if not self.full.ensure(total):
            raise OracleNoMem(total)
        fp = self.full.take(total)
        build = extend_slots_three_part if three_part else extend_slots_plain
        full_out, swa_out = [], []
        off = 0
        for r in range(len(pre)):
            full_out += build(pre[r], seq[r], last[r], fp[off:off + deltas[r]], ps)
            off += deltas[r]
            swa_out += [ring_slot(reqs[r], t, self.ring_size, ps) for t in range(pre[r], seq[r])]
        for f, s in zip(full_out, swa_out):
            self.mapping[f] = s
        return full_out, swa_out

    def alloc_decode(self, seq_lens, last_loc, req_idx=None):
        seq = [int(x) for x in seq_lens]
        return self.alloc_extend([s - 1 for s in seq], seq, last_loc, req_idx)

    def free_swa(self, full_idx) -> None:
        for i in full_idx:
            self.mapping[int(i)] = 0

    def check_no_duplicate_pages(self) -> None:
        pages = self.full.all_free_pages()
        assert len(pages) == len(set(pages)), "duplicate free page"
        assert all(1 <= p <= self.full.num_pages for p in pages)
