"""Pins of the oracle's SWA radix component ([SWA note], "prefix cache:
tombstones and the window hit rule").

- a scripted scenario whose expected matches, tombstones and releases are
  worked out by hand from the page's rules;
- the match end against the direct statement of the hit rule (all of the
  min(e, W) tokens before e live) and maximality over page boundaries;
- conservation: every inserted slot is cached or released, never both, never
  twice; no tombstone leaf; locked prefixes survive any eviction.
"""
import random

import pytest

from oracle import hitrule as H
from oracle.radix import RadixSWA


def test_scripted_scenario():
    R = RadixSWA(page_size=1, window=2)
    R.insert([1, 2, 3, 4, 5, 6], [10, 11, 12, 13, 14, 15], swa_evicted=0)
    assert R.take_releases() == ([], [])
    e, slots, nid = R.match([1, 2, 3, 4, 9])
    assert (e, slots) == (4, [10, 11, 12, 13])           # diverges after 4: node split there
    # SWA eviction of 3 tokens: LRU by last use - the unmatched tail [5, 6] is
    # older than the matched head, and it is a leaf, so it is deleted whole.
    assert R.evict_swa(2) == 2
    assert R.take_releases() == ([14, 15], [])
    # now [1..4] is a leaf: SWA-evicting it deletes it (no tombstone leaf)
    assert R.evict_swa(1) == 4
    assert R.take_releases() == ([10, 11, 12, 13], [])
    assert R.cached_tokens() == 0
    # A request whose first 4 tokens lost their SWA KV goes in as a
    # tombstone prefix followed by live tokens.
    R.insert([1, 2, 3, 4, 5, 6, 7], [20, 21, 22, 23, 24, 25, 26], swa_evicted=4)
    R.check()
    e, slots, _ = R.match([1, 2, 3, 4, 5, 6, 7, 8])
    assert (e, slots) == (7, [20, 21, 22, 23, 24, 25, 26])   # 2 live tokens before 7
    e, _, _ = R.match([1, 2, 3, 4, 5])
    assert e == 0                                             # only 1 live token before 5
    e, _, _ = R.match([1, 2, 3, 4, 5, 6])
    assert e == 6
    # A new request with live SWA KV over the tombstone prefix revives it:
    # the node takes the new slots, its old ones are released; the duplicate
    # tail of the new request is released.
    R.insert([1, 2, 3, 4, 5], [30, 31, 32, 33, 34], swa_evicted=0)
    assert R.take_releases() == ([20, 21, 22, 23, 34], [])
    e, slots, _ = R.match([1, 2, 3, 4, 5, 6, 7])
    assert (e, slots) == (7, [30, 31, 32, 33, 24, 25, 26])
    # A request that took its prefix from the tree hands it back unchanged:
    # only its own new tokens are added, nothing is released.
    e, slots, _ = R.match([1, 2, 3, 4, 5, 6])
    R.insert([1, 2, 3, 4, 5, 6, 8, 8], slots + [50, 51], swa_evicted=0)
    assert R.take_releases() == ([], [])
    # An inserted request evicted everywhere adds no tombstone leaf.
    R.insert([9, 9, 9], [40, 41, 42], swa_evicted=3)
    assert R.take_releases() == ([40, 41, 42], [])
    R.check()


def _random_ops(seed, ps, W, n_ops=300):
    rnd = random.Random(seed)
    R = RadixSWA(ps, W)
    vocab = [1, 2, 3]
    next_slot = [100]
    history = []
    inserted, freed_full, freed_swa = set(), [], []
    locks = []
    for _ in range(n_ops):
        op = rnd.random()
        if op < 0.35 or not history:
            base = rnd.choice(history) if history and rnd.random() < 0.7 else []
            cut = rnd.randint(0, len(base))
            toks = base[:cut] + [rnd.choice(vocab) for _ in range(rnd.randint(1, 6) * ps)]
            n = (len(toks) // ps) * ps
            slots = list(range(next_slot[0], next_slot[0] + n))
            next_slot[0] += n
            ev = rnd.randint(0, n // ps) * ps
            R.insert(toks, slots, ev)
            inserted.update(slots)
            history.append(toks)
        elif op < 0.65:
            q = rnd.choice(history)[: rnd.randint(0, 40)] + [rnd.choice(vocab)]
            e, slots, nid = R.match(q)
            yield ("match", q, e, slots, R)
            if rnd.random() < 0.3 and e > 0:
                locks.append((nid, R.lock(nid)))
        elif op < 0.8:
            R.evict_swa(rnd.randint(1, 3 * ps))
        elif op < 0.9:
            R.evict_full(rnd.randint(1, 3 * ps))
        elif locks:
            nid, span = locks.pop(rnd.randrange(len(locks)))
            R.unlock(nid, span)
        f, s = R.take_releases()
        freed_full += f
        freed_swa += s
        cached = R.check()
        assert len(freed_full) == len(set(freed_full))
        assert len(freed_swa) == len(set(freed_swa))
        assert not (cached & set(freed_full))
        assert cached | set(freed_full) == inserted
        for nid, _ in locks:                 # locked prefixes stay cached
            assert nid in R.nodes
    assert all(nd.full_lock == 0 and nd.swa_lock == 0 for nd in R.nodes.values()) or locks


@pytest.mark.parametrize("ps,W", [(1, 2), (1, 5), (2, 3), (4, 4)])
def test_match_end_is_the_hit_rule(ps, W):
    for ev in _random_ops(ps * 10 + W, ps, W):
        _, q, e, slots, R = ev
        assert e % ps == 0 and len(slots) == e
        # re-walk the cached path of q to read the tombstone flags
        flags, node, pos = [], R.root, 0
        n = (len(q) // ps) * ps
        while pos < n:
            ch = node.children.get(tuple(q[pos:pos + ps]))
            if ch is None:
                break
            c = 0
            while c < len(ch.key) and pos + c < n and ch.key[c:c + ps] == q[pos + c:pos + c + ps]:
                c += ps
            flags += [ch.tomb] * c
            pos += c
            if c < len(ch.key):
                break
            node = ch
        assert H.usable_brute(flags, e, W)
        for e2 in range(e + ps, pos + 1, ps):
            assert not H.usable_brute(flags, e2, W)


def test_locked_prefix_survives_eviction():
    R = RadixSWA(page_size=2, window=4)
    R.insert(list(range(12)), list(range(100, 112)), 0)
    R.insert(list(range(6)) + [50, 51], [200 + i for i in range(8)], 0)
    R.take_releases()
    e, slots, nid = R.match(list(range(10)))
    assert e == 10
    span = R.lock(nid)
    R.evict_full(10 ** 6)
    R.evict_swa(10 ** 6)
    e2, slots2, _ = R.match(list(range(10)))
    assert (e2, slots2) == (10, slots)         # full path kept, last W tokens live
    R.unlock(nid, span)
    assert all(nd.full_lock == 0 and nd.swa_lock == 0 for nd in R.nodes.values())
    R.evict_full(10 ** 6)
    assert R.cached_tokens() == 0
