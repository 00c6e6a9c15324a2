"""Pins of the oracle's per-request SWA ring against the pages and against
the paged two-pool oracle ("SGLang source teardown (15)", section "why
sliding windows can be accounted per request").

- the capacity rule the pages print: one ring per request slot, each ring
  rounded up to whole pages;
- brute force: while requests grow by decode steps and chunks, the ring slots
  of every live window are distinct, inside their own ring, and disjoint
  between requests;
- the full-pool side is exactly the paged allocator's full side;
- attention read through the ring tables equals attention read through the
  paged tables on the same stored KV (the ring changes where keys live, never
  which keys a query sees);
- the misuse cases the reading rejects.
"""
import random

import numpy as np
import pytest

from oracle import allocator as OA
from oracle import attention as OT
from oracle import kvstore as OK


def test_capacity_rule_from_the_pages():
    # cost = ceil(ring_size / ps) * ps; size_swa = slots * cost
    assert OA.ring_cost(128, 64) == 128
    assert OA.ring_cost(129, 64) == 192
    assert OA.ring_cost(16, 1) == 16
    assert OA.ring_pool_size(48, 128, 64) == 48 * 128
    assert OA.ring_pool_size(7, 130, 16) == 7 * 144
    # every slot of every ring is distinct and past the padding page
    ps, ring, n = 4, 10, 5
    slots = {OA.ring_slot(r, t, ring, ps) for r in range(n) for t in range(OA.ring_cost(ring, ps))}
    assert len(slots) == n * OA.ring_cost(ring, ps)
    assert min(slots) == ps and max(slots) == ps + OA.ring_pool_size(n, ring, ps) - 1


def _grow(alloc, rt, lens, r, new_len, ps):
    pre = lens.get(r, 0)
    last = int(rt[r, pre - 1]) if pre else -1
    if isinstance(alloc, OA.RingTwoPoolAllocator):
        f, s = alloc.alloc_extend([pre], [new_len], [last], [r])
    else:
        f, s = alloc.alloc_extend([pre], [new_len], [last])
    rt[r, pre:new_len] = f
    lens[r] = new_len
    return f, s


@pytest.mark.parametrize("ps,ring,wx", [(1, 9, 6), (4, 13, 7), (16, 40, 15)])
def test_live_windows_never_collide(ps, ring, wx):
    rnd = random.Random(ps * 100 + ring)
    slots_n, max_ctx = 5, 400
    A = OA.RingTwoPoolAllocator(ps * 600, ps, ring, slots_n, wx)
    rt = np.zeros((slots_n, max_ctx), np.int64)
    lens = {}
    for _ in range(200):
        r = rnd.randrange(slots_n)
        pre = lens.get(r, 0)
        step = rnd.randint(1, A.cost - wx)
        if pre + step > max_ctx:
            continue
        _grow(A, rt, lens, r, pre + step, ps)
        # every live window (last wx+1 positions of each request) is intact
        seen = {}
        for q, n in lens.items():
            for t in range(max(0, n - 1 - wx), n):
                s = A.translate(int(rt[q, t]))
                assert s == OA.ring_slot(q, t, ring, ps)
                lo = ps + q * A.cost
                assert lo <= s < lo + A.cost
                assert s not in seen, (q, t, seen.get(s))
                seen[s] = (q, t)


def test_full_side_matches_paged_allocator():
    ps, wx = 4, 7
    ring_alloc = OA.RingTwoPoolAllocator(ps * 64, ps, 16, 4, wx)
    paged = OA.TwoPoolAllocator(ps * 64, ps * 64, ps)
    rt_a = np.zeros((4, 200), np.int64)
    rt_b = np.zeros((4, 200), np.int64)
    la, lb = {}, {}
    rnd = random.Random(3)
    for _ in range(40):
        r = rnd.randrange(4)
        n = la.get(r, 0) + rnd.randint(1, 9)
        if n > 200:
            continue
        fa, _ = _grow(ring_alloc, rt_a, la, r, n, ps)
        fb, _ = _grow(paged, rt_b, lb, r, n, ps)
        assert fa == fb
    assert ring_alloc.full.free == paged.full.free


def test_attention_through_ring_equals_paged():
    ps, wx, ring = 4, 7, 12
    layers = [(OT.SLIDING, wx, 2), (OT.FULL, 0, 2)]
    D, Hq, B = 8, 4, 3
    rng = np.random.default_rng(5)
    ring_alloc = OA.RingTwoPoolAllocator(ps * 64, ps, ring, B, wx)
    paged = OA.TwoPoolAllocator(ps * 64, ps * 64, ps)
    pools_r = OK.OraclePools(layers, ps * 64, ring_alloc.size_swa, ps, D, "f32")
    pools_p = OK.OraclePools(layers, ps * 64, ps * 64, ps, D, "f32")
    rt_r = np.zeros((B, 200), np.int64)
    rt_p = np.zeros((B, 200), np.int64)
    lr, lp = {}, {}
    for step in range(12):
        for b in range(B):
            n = lr.get(b, 0) + (1 + (b + step) % (ring - wx))
            fr, sr = _grow(ring_alloc, rt_r, lr, b, n, ps)
            fp, sp = _grow(paged, rt_p, lp, b, n, ps)
            k = rng.standard_normal((len(fr), 2, D)).astype(np.float32)
            v = rng.standard_normal((len(fr), 2, D)).astype(np.float32)
            for l in range(2):
                pools_r.store(l, k, v, fr, sr)
                pools_p.store(l, k, v, fp, sp)
        pos = [(b, lr[b] - 1) for b in range(B)]
        q = rng.standard_normal((B, Hq, D))
        sinks = rng.standard_normal(Hq)
        for l in range(2):
            o_r = OK.attention_through_tables(pools_r, ring_alloc, l, rt_r, list(range(B)), pos, q,
                                              sinks, 0.35)
            o_p = OK.attention_through_tables(pools_p, paged, l, rt_p, list(range(B)), pos, q,
                                              sinks, 0.35)
            np.testing.assert_array_equal(o_r, o_p)


def test_eviction_and_free_only_clear_the_mapping():
    ps, wx = 4, 7
    A = OA.RingTwoPoolAllocator(ps * 64, ps, 16, 2, wx)
    rt = np.zeros((2, 100), np.int64)
    lens = {}
    for n in (9, 18, 27):
        _grow(A, rt, lens, 0, n, ps)
    before = A.available_size()
    ev, freed = OA.evict_swa(A, rt, [0], [27], [0], [0], wx, 0)
    assert freed == 0 and A.available_size() == before
    old, new = 0, ev[0]
    assert new == ((27 - wx) // ps) * ps
    assert all(A.translate(int(rt[0, t])) == 0 for t in range(old, new))
    assert all(A.translate(int(rt[0, t])) > 0 for t in range(new, 27))
    A.free([int(x) for x in rt[0, :27]])
    assert A.available_size() == ps * 64
    assert all(A.translate(int(rt[0, t])) == 0 for t in range(27))
    A.check_no_duplicate_pages()


def test_rejected_cases():
    with pytest.raises(ValueError):
        OA.RingTwoPoolAllocator(64, 4, 7, 2, 7)          # ring smaller than W
    A = OA.RingTwoPoolAllocator(256, 4, 16, 2, 7)
    with pytest.raises(ValueError):
        A.alloc_extend([0], [10], [-1], [0])              # 10 new + 7 lookback > 16
    with pytest.raises(ValueError):
        A.alloc_extend([0], [4], [-1], [2])               # no ring for slot 2
    with pytest.raises(ValueError):
        A.alloc(4)
    rt = np.zeros((2, 400), np.int64)
    lens = {}
    with pytest.raises(OA.OracleNoMem):
        for i in range(100):
            _grow(A, rt, lens, i % 2, lens.get(i % 2, 0) + 9, 4)
