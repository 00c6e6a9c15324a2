"""Pins of the unified-pool oracle (FULL and SWA allocated from the two ends
of one page range; [Pools 15], allocator-family table,
UnifiedSWATokenToKVPoolAllocator; [PR 34602], multi_ended_allocator.py).

* a hand-worked sequence (pages, frontiers, gap, tombstones, kernel ids);
* with no release, the unified pool is the two-pool allocator whose FULL
  ledger starts at 1, 2, ... and whose SWA ledger starts at P, P-1, ...: the
  FULL physical slots equal the two-pool full slots and the SWA physical
  slots equal the two-pool mapping (the shared ids replace the table);
* NOMEM leaves every list, frontier and table as it was;
* random operation sequences keep every page owned exactly once (FULL below
  its frontier, SWA above its own, the rest in the gap), never hand out a
  page twice, and ``available_size`` equals a brute-force search for the
  largest allocation that succeeds."""
import copy
import random

import pytest

from oracle import allocator as OA
from oracle import envelope as OE
from oracle import unified as OU


def test_hand_worked_sequence():
    U = OU.MultiEndedPool(8, 2)
    # request 0: tokens 0..2 (two virtual pages), request 1: tokens 0..1 (one)
    virt = U.alloc_extend([0, 0], [3, 2], [-1, -1])
    assert virt == [2, 3, 4, 6, 7]                      # virtual pages 1, 2, 3
    assert U.v2p[OU.FULL][1:4] == [1, 2, 3]             # low end, upward
    assert U.v2p[OU.SWA][1:4] == [8, 7, 6]              # high end, downward
    assert (U.low, U.high, U.gap()) == (3, 6, 2)
    # kernel ids of one layer (2 row blocks per page): phys * 4 + t % 2
    assert OE.translate_for_kernel(U.v2p[OU.FULL], virt, 2, 2) == [4, 5, 8, 12, 13]
    assert OE.translate_for_kernel(U.v2p[OU.SWA], virt, 2, 2) == [32, 33, 28, 24, 25]
    # request 0 continues inside its open page (token 3 after slot 4), then a new page
    assert U.alloc_extend([3], [5], [4]) == [5, 8]      # virtual page 4
    assert (U.v2p[OU.FULL][4], U.v2p[OU.SWA][4]) == (4, 5)
    assert U.gap() == 0
    assert U.available_size() == 0
    with pytest.raises(OU.UnifiedNoMem):
        U.alloc_extend([0], [1], [-1])
    # SWA page of virtual page 1 released: not at the frontier, so it stays
    # in the SWA released set; the page's kernel ids clamp to the sink
    U.free_swa([2, 3])
    assert U.v2p[OU.SWA][1] == -1 and U.released[OU.SWA] == [8]
    assert OE.translate_for_kernel(U.v2p[OU.SWA], [2, 3], 2, 2) == [0, 0]
    # request 1 ends: its SWA page 6 is not at the frontier (5 is), its FULL
    # page 3 is not at the frontier (4 is): both wait in their released sets
    U.free([6, 7])
    assert U.released[OU.SWA] == [6, 8] and U.released[OU.FULL] == [3]
    assert U.vfree == [3, 5, 6, 7, 8]
    # request 0 ends: FULL 1, 2, 4 released, the frontier retracts to 0; SWA
    # 7 and 5 released, the frontier retracts over 5, 6, 7, 8
    U.free([2, 3, 4, 5, 8])
    assert (U.low, U.high, U.gap()) == (0, 9, 8)
    assert U.released[OU.FULL] == [] and U.released[OU.SWA] == []
    assert U.vfree == [1, 2, 4, 3, 5, 6, 7, 8]
    U.check()


def test_reuse_nearest_own_end_first():
    """Released pages are reused from each side's own end: FULL takes its
    lowest released page, SWA its highest, before touching the gap."""
    U = OU.MultiEndedPool(12, 1)
    virt = U.alloc_extend([0, 0, 0], [3, 1, 1], [-1, -1, -1])   # 5 virtual pages
    assert U.v2p[OU.FULL][1:6] == [1, 2, 3, 4, 5]
    assert U.v2p[OU.SWA][1:6] == [12, 11, 10, 9, 8]
    U.free(virt[1:2] + virt[3:4])           # virtual pages 2 and 4: FULL 2, 4; SWA 11, 9
    assert U.released[OU.FULL] == [2, 4] and U.released[OU.SWA] == [9, 11]
    assert U.vfree[:2] == [2, 4]
    out = U.alloc_extend([0], [3], [-1])    # three pages: two reused, one from each frontier
    assert out == [2, 4, 6]
    assert [U.v2p[OU.FULL][v] for v in (2, 4, 6)] == [2, 4, 6]
    assert [U.v2p[OU.SWA][v] for v in (2, 4, 6)] == [11, 9, 7]
    U.check()


def test_no_release_reduces_to_the_two_pool_allocator():
    P, ps = 40, 4
    U = OU.MultiEndedPool(P, ps)
    T = OA.TwoPoolAllocator(P * ps, P * ps, ps, init_full=list(range(1, P + 1)),
                            init_swa=list(range(P, 0, -1)))
    rnd = random.Random(3)
    lens = {}
    for _ in range(25):
        rows = rnd.sample(range(6), 2)
        pre = [lens.get(r, 0) for r in rows]
        seq = [p + rnd.randint(0, 9) for p in pre]
        need = sum(OA.ceil_div(s, ps) - OA.ceil_div(p, ps) for p, s in zip(pre, seq))
        if not U.fits(need):
            break
        last = [lens.get((r, "last"), -1) for r in rows]
        virt = U.alloc_extend(pre, seq, last)
        full, swa = T.alloc_extend(pre, seq, last)
        assert [U.physical_slot(OU.FULL, t) for t in virt] == full
        assert [U.physical_slot(OU.SWA, t) for t in virt] == swa
        assert virt == full                  # identity FULL table while nothing is released
        off = 0
        for r, p, s in zip(rows, pre, seq):
            if s > p:
                lens[(r, "last")] = virt[off + s - p - 1]
            off += s - p
            lens[r] = s
    U.check()


def test_nomem_changes_nothing():
    U = OU.MultiEndedPool(6, 1)
    U.alloc_extend([0], [2], [-1])                   # FULL 1, 2; SWA 6, 5; gap of 2
    before = copy.deepcopy(U.__dict__)
    with pytest.raises(OU.UnifiedNoMem):
        U.alloc_extend([0, 0], [1, 1], [-1, -1])     # needs 2 pages on each side
    assert U.__dict__ == before


@pytest.mark.parametrize("ps,P,seed", [(1, 48, 0), (4, 40, 1), (16, 24, 2)])
def test_random_sequences_conserve_pages(ps, P, seed):
    rnd = random.Random(seed)
    U = OU.MultiEndedPool(P, ps)
    rt = {}
    evicted = {}
    for step in range(300):
        op = rnd.random()
        live = sorted(rt)
        if op < 0.5 or not live:
            rows = rnd.sample(range(8), rnd.randint(1, 3))
            pre = [len(rt.get(r, [])) for r in rows]
            seq = [p + rnd.randint(0, 2 * ps + 2) for p in pre]
            need = sum(OA.ceil_div(s, ps) - OA.ceil_div(p, ps) for p, s in zip(pre, seq))
            # brute force: the largest whole-page allocation that succeeds
            n_ok = 0
            while True:
                trial = copy.deepcopy(U)
                try:
                    trial.alloc_extend([0], [(n_ok + 1) * ps], [-1])
                except OU.UnifiedNoMem:
                    break
                n_ok += 1
            assert U.available_size() == n_ok * ps
            last = [rt[r][-1] if rt.get(r) else -1 for r in rows]
            if U.fits(need):
                virt = U.alloc_extend(pre, seq, last)
                off = 0
                for r, p, s in zip(rows, pre, seq):
                    rt.setdefault(r, []).extend(virt[off:off + s - p])
                    off += s - p
                    evicted.setdefault(r, 0)
            else:
                with pytest.raises(OU.UnifiedNoMem):
                    U.alloc_extend(pre, seq, last)
        elif op < 0.7:
            r = rnd.choice(live)
            U.free(rt.pop(r))
            evicted.pop(r, None)
        elif op < 0.9:
            r = rnd.choice(live)
            ev = OU.evict_swa(U, {r: rt[r]}, [r], [len(rt[r])], [evicted[r]], [0],
                              rnd.choice([1, 3, 7]), 0)
            evicted[r] = ev[0]
        else:
            # free_swa of a page-aligned stretch, then a full free later must
            # not release those SWA pages twice
            r = rnd.choice(live)
            k = (len(rt[r]) // ps) * ps
            if k > evicted[r]:
                U.free_swa(rt[r][evicted[r]:k])
                evicted[r] = k
        U.check()
    for r in list(rt):
        U.free(rt.pop(r))
    U.check()
    assert (U.low, U.high) == (0, P + 1) and len(U.vfree) == P
