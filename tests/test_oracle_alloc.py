"""Pins of the oracle's allocator against the closed forms, invariants and
brute force the pages fix (two-pool allocator, paged ledgers, eviction)."""
import random

import numpy as np
import pytest

from oracle import allocator as O
from oracle.allocator import ceil_div


# ------------------------------------------------------------------ slots ---
@pytest.mark.parametrize("ps", [1, 2, 4, 16, 64])
def test_two_statements_of_extend_agree(ps):
    rnd = random.Random(ps)
    for _ in range(300):
        pre = rnd.randrange(0, 5 * ps + 3)
        seq = pre + rnd.randrange(0, 6 * ps + 3)
        n_new = ceil_div(seq, ps) - ceil_div(pre, ps)
        pages = rnd.sample(range(1, 1000), n_new)
        last = (rnd.randrange(1, 900) * ps + (pre - 1) % ps) if pre > 0 else -1
        a = O.extend_slots_plain(pre, seq, last, pages, ps)
        b = O.extend_slots_three_part(pre, seq, last, pages, ps)
        assert a == b
        assert len(a) == seq - pre


@pytest.mark.parametrize("ps", [1, 4, 64])
def test_extend_closed_forms(ps):
    """slot(p, k) = p * ps + k; page counts are ceil differences; every new
    page is used; offsets inside a page follow the position."""
    rnd = random.Random(7 + ps)
    for _ in range(200):
        pre = rnd.randrange(0, 4 * ps + 2)
        seq = pre + rnd.randrange(1, 5 * ps + 2)
        n_new = ceil_div(seq, ps) - ceil_div(pre, ps)
        last = (rnd.randrange(500, 900) * ps + (pre - 1) % ps) if pre > 0 else -1
        pages = rnd.sample(range(1, 500), n_new)
        out = O.extend_slots_plain(pre, seq, last, pages, ps)
        for t, s in zip(range(pre, seq), out):
            assert s % ps == t % ps
        used = sorted(set(s // ps for s in out) - ({last // ps} if pre % ps else set()))
        assert used == sorted(pages)


def test_sentinel_translates_minus_one():
    a = O.TwoPoolAllocator(64, 32, 4)
    assert len(a.mapping) == 64 + 4 + 1
    assert a.translate(-1) == -1
    assert all(m == 0 for m in a.mapping[:-1])
    full, swa = a.alloc_extend([0], [5], [-1])
    assert len(full) == len(swa) == 5
    assert a.translate(full) == swa


def test_available_is_min_of_pools():
    a = O.TwoPoolAllocator(256, 64, 4)
    assert a.available_size() == 64
    a.alloc_extend([0, 0], [10, 7], [-1, -1])          # 3 + 2 pages each side
    assert a.full.available_size() == 256 - 20
    assert a.swa.available_size() == 64 - 20
    assert a.available_size() == 44


def test_nomem_leaves_state_unchanged():
    a = O.TwoPoolAllocator(256, 32, 4)
    a.alloc_extend([0], [9], [-1])
    before = (list(a.full.free), list(a.swa.free), list(a.mapping))
    with pytest.raises(O.OracleNoMem):
        a.alloc_extend([0], [40], [-1])                 # SWA pool short
    assert (list(a.full.free), list(a.swa.free), list(a.mapping)) == before


def test_free_prepends_unique_sorted_pages():
    led = O.PageLedger(64, 4)
    taken = led.take(10)
    rest = list(led.free)
    slots = [p * 4 + k for p in reversed(taken[:5]) for k in (3, 0, 1)]
    led.free_slots(slots)
    assert led.free == list(np.unique(np.array(slots) // 4)) + rest


def test_need_sort_stages_then_merges_sorted():
    led = O.PageLedger(64, 4, need_sort=True)
    t = led.take(16)                                    # all pages
    led.free_slots([t[5] * 4, t[2] * 4 + 1])
    led.free_slots([t[9] * 4 + 3])
    assert led.free == [] and led.available_size() == 3 * 4
    assert led.ensure(2)
    assert led.free == sorted([t[5], t[2], t[9]]) and led.staged == []


def test_two_step_free_is_double_free_safe():
    rnd = random.Random(3)
    for ps in (1, 4, 16):
        a = O.TwoPoolAllocator(ps * 100, ps * 60, ps)
        full, swa = a.alloc_extend([0, 0], [ps * 7 + 1, ps * 3 + 2], [-1, -1])
        n0 = len(full)
        r0 = full[:ps * 7 + 1]
        # free_swa on a prefix first (eviction), then the whole request.
        k = ps * 4
        a.free_swa(r0[:k])
        assert all(a.translate(f) == 0 for f in r0[:k])
        a.free(r0)
        a.free(full[ps * 7 + 1:])
        a.check_no_duplicate_pages()
        assert a.full.available_size() == ps * 100
        assert a.swa.available_size() == ps * 60
        # and in the other order nothing is freed twice either
        full, _ = a.alloc_extend([0], [ps * 5], [-1])
        a.free(full)
        a.free_swa(full)
        a.check_no_duplicate_pages()
        assert a.swa.available_size() == ps * 60


def test_swa_offsets_follow_full_offsets():
    a = O.TwoPoolAllocator(64 * 40, 64 * 30, 64)
    full, swa = a.alloc_extend([0, 0, 0], [100, 64, 3], [-1, -1, -1])
    assert all(f % 64 == s % 64 for f, s in zip(full, swa))
    last = [full[99], full[100 + 63], full[-1]]
    f2, s2 = a.alloc_decode([101, 65, 4], last)
    assert all(f % 64 == s % 64 for f, s in zip(f2, s2))
    assert f2[0] == full[99] + 1 and f2[2] == full[-1] + 1
    assert f2[1] % 64 == 0                               # crossed into a new page


# --------------------------------------------------------- brute force ---
@pytest.mark.parametrize("ps,need_sort", [(1, False), (2, False), (4, True), (4, False)])
def test_random_sequences_keep_invariants(ps, need_sort):
    """Brute-force model on small pools: slots never shared, pages conserved,
    mapping consistent, and NOMEM exactly when pages are short."""
    rnd = random.Random(11 * ps + need_sort)
    nf, ns = ps * 24, ps * 12
    a = O.TwoPoolAllocator(nf, ns, ps, need_sort)
    reqs = {}            # rid -> list of full slots (position order)
    evicted = {}
    for step in range(400):
        op = rnd.random()
        if op < 0.45 or not reqs:
            # extend a batch of 1..3 requests (new or existing)
            batch = []
            for _ in range(rnd.randint(1, 3)):
                if reqs and rnd.random() < 0.6:
                    rid = rnd.choice(sorted(reqs))
                else:
                    rid = max(list(reqs) + [0]) + 1
                if rid in [b[0] for b in batch]:
                    continue
                batch.append((rid, rnd.randint(0, 3 * ps)))
            pre = [len(reqs.get(r, [])) for r, _ in batch]
            seq = [p + e for p, (_, e) in zip(pre, batch)]
            last = [reqs[r][-1] if reqs.get(r) else -1 for r, _ in batch]
            need = sum(ceil_div(s, ps) - ceil_div(p, ps) for p, s in zip(pre, seq))
            free_f = a.full.available_size() // ps
            free_s = a.swa.available_size() // ps
            try:
                full, swa = a.alloc_extend(pre, seq, last)
            except O.OracleNoMem:
                assert need > min(free_f, free_s)
                continue
            assert need <= min(free_f, free_s)
            off = 0
            for (rid, e), p in zip(batch, pre):
                reqs.setdefault(rid, []).extend(full[off:off + e])
                evicted.setdefault(rid, 0)
                off += e
        elif op < 0.7:
            rid = rnd.choice(sorted(reqs))
            a.free(reqs.pop(rid))
            evicted.pop(rid, None)
        else:
            # evict SWA of the oldest tokens of one request (page aligned)
            rid = rnd.choice(sorted(reqs))
            L = len(reqs[rid])
            wx = rnd.randint(1, 2 * ps)
            old, new = O.evict_range(L, evicted[rid], 0, wx, ps, 0)
            if new > old:
                a.free_swa(reqs[rid][old:new])
                evicted[rid] = new
        a.check_no_duplicate_pages()
        # Conservation: free pages + pages held by live requests = all pages.
        held_full = set(s // ps for r in reqs.values() for s in r)
        held_swa = set(a.translate(s) // ps for r in reqs.values() for s in r
                       if a.translate(s) > 0)
        assert len(held_full) + a.full.available_size() // ps == nf // ps
        assert len(held_swa) + a.swa.available_size() // ps == ns // ps
        # No slot is owned twice.
        allslots = [s for r in reqs.values() for s in r]
        assert len(allslots) == len(set(allslots))
        live_swa = [a.translate(s) for s in allslots if a.translate(s) > 0]
        assert len(live_swa) == len(set(live_swa))
        # Evicted prefixes map to 0, the rest to live slots.
        for rid, r in reqs.items():
            for t, s in enumerate(r):
                assert (a.translate(s) == 0) == (t < evicted[rid])


# -------------------------------------------------------------- eviction ---
def test_evict_range_worked_examples():
    # Chunked prefill of the extend workload: 24K cached prefix, window 128
    # (127 prior keys), page 64: SWA KV below floor((24576-127)/64)*64 goes.
    assert O.evict_range(24576, 0, 0, 127, 64, 0) == (0, 24448)
    # Radix bound uses max(W, page).
    assert O.evict_range(24576, 0, 0, 15, 64, 0, radix=True) == (0, 24512)
    # Decode: fires only when >= interval tokens slid out past 'evicted'.
    assert O.evict_range(24448 + 127 + 127, 24448, 0, 127, 64, 128) == (24448, 24448)
    assert O.evict_range(24448 + 127 + 128, 24448, 0, 127, 64, 128) == (24448, 24576)
    # Protected prefix is rounded up to a page before freeing.
    assert O.evict_range(1000, 0, 70, 127, 64, 0) == (128, 832)


def test_eviction_keeps_every_window_key_live():
    """After each pass the next query's window maps to live SWA slots and the
    pages freed are (new - old) / ps."""
    from oracle import attention as A
    ps, wx = 4, 7
    a = O.TwoPoolAllocator(ps * 64, ps * 12, ps)
    rt = np.zeros((3, 200), np.int64)
    lens = [0, 0]
    ev = [0, 0]
    for step in range(60):
        pre = list(lens)
        seq = [l + (5 if step < 4 else 1) for l in lens]
        ev2, freed = O.evict_swa(a, rt, [1, 2], pre, ev, [0, 0], wx, 0 if step < 4 else 3)
        assert freed == sum((n - o) // ps for o, n in zip(ev, ev2))
        ev = ev2
        last = [rt[1 + b, pre[b] - 1] if pre[b] else -1 for b in range(2)]
        full, _ = a.alloc_extend(pre, seq, last)
        off = 0
        for b in range(2):
            n = seq[b] - pre[b]
            rt[1 + b, pre[b]:seq[b]] = full[off:off + n]
            off += n
            for p in range(pre[b], seq[b]):
                for j in A.key_positions(A.SLIDING, wx, p):
                    assert a.translate(int(rt[1 + b, j])) > 0
        lens = seq
    a.check_no_duplicate_pages()
