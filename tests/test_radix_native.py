"""The native SWA radix tree (host C++ in libswa) against the oracle tree on
random operation sequences: every match (end, slots, node), every release
list, every eviction count and the cached / live sizes, identical.  Host
code only: runs without a GPU."""
import random

import pytest

from oracle.radix import RadixSWA

api = pytest.importorskip("hybrid_sliding_window_gb300.api")


def _lib_or_skip():
    try:
        api.lib()
    except Exception as e:  # library not built here
        pytest.skip(f"libswa not loadable: {e}")


@pytest.mark.parametrize("ps,W,seed", [(1, 2, 0), (1, 7, 1), (2, 3, 2), (4, 4, 3), (4, 9, 4),
                                       (16, 31, 5)])
def test_native_tree_matches_oracle(ps, W, seed):
    _lib_or_skip()
    rnd = random.Random(seed)
    O = RadixSWA(ps, W)
    N = api.RadixSWA(ps, W)
    vocab = [1, 2, 3]
    history = []
    slot = 1000
    locks = []
    for step in range(600):
        op = rnd.random()
        if op < 0.35 or not history:
            base = rnd.choice(history) if history and rnd.random() < 0.7 else []
            toks = base[:rnd.randint(0, len(base))] + [rnd.choice(vocab) for _ in
                                                        range(rnd.randint(1, 6) * ps + rnd.randint(0, ps - 1))]
            n = len(toks)
            slots = list(range(slot, slot + n))
            slot += n
            ev = rnd.randint(0, n // ps) * ps
            O.insert(toks, slots, ev)
            N.insert(toks, slots, ev)
            history.append(toks)
        elif op < 0.65:
            q = rnd.choice(history)[: rnd.randint(0, 60)] + [rnd.choice(vocab)]
            a = O.match(q)
            b = N.match(q)
            assert a == b, (step, a, b)
            if rnd.random() < 0.25:
                # a request that took its prefix from the tree finishes
                toks = q[:a[0]] + [rnd.choice(vocab) for _ in range(rnd.randint(0, 3) * ps)]
                extra = len(toks) - a[0]
                slots_r = a[1] + list(range(slot, slot + extra))
                slot += extra
                ev = rnd.randint(0, len(toks) // ps) * ps
                O.insert(toks, slots_r, ev)
                N.insert(toks, slots_r, ev)
                history.append(toks)
            elif a[0] > 0 and rnd.random() < 0.3:
                sa, sb = O.lock(a[2]), N.lock(b[2])
                assert sa == sb
                locks.append((a[2], sa))
        elif op < 0.8:
            k = rnd.randint(1, 3 * ps)
            assert O.evict_swa(k) == N.evict(k, swa_only=True)
        elif op < 0.9:
            k = rnd.randint(1, 3 * ps)
            assert O.evict_full(k) == N.evict(k)
        elif locks:
            nid, span = locks.pop(rnd.randrange(len(locks)))
            O.unlock(nid, span)
            N.unlock(nid, span)
        of, osw = O.take_releases()
        nf, live, nsw = N.releases()
        assert of == nf.tolist() and osw == nsw.tolist(), step
        assert (O.cached_tokens(), O.live_tokens()) == N.sizes()[:2]
        assert len(O.nodes) - 1 == N.sizes()[2]


def test_native_tree_rejections():
    _lib_or_skip()
    N = api.RadixSWA(4, 3)
    with pytest.raises(api.SwaError):
        N.insert([1, 2, 3, 4], [1, 2, 3, 4], swa_evicted=2)     # not a page multiple
    with pytest.raises(api.SwaError):
        N.unlock(0 + 12345, 0)                                   # unknown node
    N.insert([1, 2, 3, 4], [5, 6, 7, 8], 0)
    e, _, node = N.match([1, 2, 3, 4])
    span = N.lock(node)
    N.unlock(node, span)
    with pytest.raises(api.SwaError):
        N.unlock(node, span)                                     # no lock left
