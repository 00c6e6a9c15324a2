"""The unified FULL/SWA pool allocated from both ends of one page range
([Pools 15], allocator-family table, UnifiedSWATokenToKVPoolAllocator;
[PR 34602], multi_ended_allocator.py) against the oracle, bit for bit:
random sequences of allocations (with req_to_token writes), frees, free_swa
of page-aligned stretches and eviction passes; after every operation the
virtual slots, req_to_token, both virtual-to-physical tables, both released
sets, the two frontiers, the virtual-id ring, the available size and the
kernel-facing ids of every live token (swa_translate_for_kernel through
each table) must equal the oracle's.  NOMEM must agree and change nothing."""
import random

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import allocator as OA  # noqa: E402
from oracle import envelope as OE  # noqa: E402
from oracle import unified as OU  # noqa: E402


class UPair:
    def __init__(self, P, ps, rows=8, ctx=256):
        self.u = api.UnifiedPool(P, ps, max_batch=8)
        self.o = OU.MultiEndedPool(P, ps)
        self.P, self.ps = P, ps
        self.rt = torch.zeros((rows + 1, ctx), dtype=torch.int32, device="cuda")
        self.ort = np.zeros((rows + 1, ctx), np.int64)

    def alloc(self, rows, pre, seq):
        n = int(sum(s - p for p, s in zip(pre, seq)))
        out = torch.empty(max(n, 1), dtype=torch.int64, device="cuda")
        d = lambda x: torch.tensor(np.asarray(x, np.int64), device="cuda")
        last = [int(self.ort[r, p - 1]) if p else -1 for r, p in zip(rows, pre)]
        try:
            want = self.o.alloc_extend(pre, seq, last)
        except OU.UnifiedNoMem:
            with pytest.raises(api.SwaNoMem):
                api.swa_unified_alloc_extend(self.u, d(pre), d(seq), None, pre, seq, out,
                                             req_to_token=self.rt, req_idx=d(rows))
            return None
        api.swa_unified_alloc_extend(self.u, d(pre), d(seq), None, pre, seq, out,
                                     req_to_token=self.rt, req_idx=d(rows))
        assert out[:n].cpu().tolist() == want
        off = 0
        for r, p, s in zip(rows, pre, seq):
            self.ort[r, p:s] = want[off:off + s - p]
            off += s - p
        return want

    def check(self):
        torch.cuda.synchronize()
        assert api.swa_unified_device_check(self.u) == 0
        o = self.o
        assert self.u.v2p(True).cpu().tolist() == o.v2p[OU.FULL]
        assert self.u.v2p(False).cpu().tolist() == o.v2p[OU.SWA]
        assert self.u.released(True) == o.released[OU.FULL]
        assert self.u.released(False) == o.released[OU.SWA]
        c = self.u.counters()
        assert (c[api.UCTR_LOW], c[api.UCTR_HIGH]) == (o.low, o.high)
        assert (c[api.UCTR_REL_FULL], c[api.UCTR_REL_SWA]) == (len(o.released[OU.FULL]),
                                                               len(o.released[OU.SWA]))
        assert self.u.virt_free() == o.vfree
        np.testing.assert_array_equal(self.rt.cpu().numpy().astype(np.int64), self.ort)
        api.swa_unified_sync(self.u)
        assert api.swa_unified_available_size(self.u) == o.available_size()
        o.check()
        # kernel-facing ids of every live token, through both tables (2 row
        # blocks per page for FULL, 6 for SWA: a 1-layer and a 3-layer envelope)
        live = [int(t) for t in self.ort.reshape(-1) if t > 0]
        if live:
            virt = torch.tensor(live, dtype=torch.int64, device="cuda")
            for side, table, mult in ((OU.FULL, self.u.v2p(True), 2),
                                      (OU.SWA, self.u.v2p(False), 6)):
                got = api.swa_translate_for_kernel(table, virt, self.ps, mult).cpu().tolist()
                assert got == OE.translate_for_kernel(o.v2p[side], live, self.ps, mult)


@pytest.mark.parametrize("ps,P,seed", [(1, 96, 0), (4, 64, 1), (16, 40, 2), (64, 33, 3)])
def test_unified_random_sequences(ps, P, seed):
    rnd = random.Random(seed)
    U = UPair(P, ps)
    lens, evicted = {}, {}
    for step in range(120):
        op = rnd.random()
        live = sorted(lens)
        if op < 0.5 or not live:
            rows = rnd.sample(range(1, 9), rnd.randint(1, 3))
            pre = [lens.get(r, 0) for r in rows]
            seq = [min(p + rnd.randint(0, 2 * ps + 3), U.rt.shape[1]) for p in pre]
            if U.alloc(rows, pre, seq) is not None:
                for r, s in zip(rows, seq):
                    lens[r] = s
                    evicted.setdefault(r, 0)
        elif op < 0.65:
            r = rnd.choice(live)
            idx = [int(x) for x in U.ort[r, :lens[r]]]
            if idx:
                api.swa_unified_free(U.u, torch.tensor(idx, dtype=torch.int64, device="cuda"))
                U.o.free(idx)
            del lens[r]
            evicted.pop(r, None)
            U.rt[r].zero_()
            U.ort[r] = 0
        elif op < 0.85:
            rows = rnd.sample(live, min(len(live), rnd.randint(1, 3)))
            pre = np.array([lens[r] for r in rows], np.int64)
            ev = np.array([evicted[r] for r in rows], np.int64)
            ev_before = ev.copy()
            wx, interval = rnd.choice([1, 3, 7]), rnd.choice([0, 2])
            ev_d = torch.tensor(ev, device="cuda")
            api.swa_unified_evict_swa(U.u, wx, U.rt, torch.tensor(rows, device="cuda"),
                                      torch.tensor(pre, device="cuda"), ev_d, pre, ev,
                                      interval=interval)
            want = OU.evict_swa(U.o, U.ort, rows, pre, ev_before, [0] * len(rows), wx, interval)
            assert ev.tolist() == want
            assert ev_d.cpu().tolist() == want
            for r, e in zip(rows, want):
                evicted[r] = e
        else:
            r = rnd.choice(live)
            k = (lens[r] // ps) * ps
            if k > evicted[r]:
                idx = [int(x) for x in U.ort[r, evicted[r]:k]]
                api.swa_unified_free_swa(U.u, torch.tensor(idx, dtype=torch.int64, device="cuda"))
                U.o.free_swa(idx)
                evicted[r] = k
        U.check()


def test_unified_fills_both_ends_then_reuses_and_retracts():
    """A hand-sized run: fill the range from both ends until NOMEM, release
    everything in an interleaved order, and end with both frontiers back at
    the ends and every page in the gap."""
    U = UPair(20, 2, ctx=64)
    rows = [1, 2, 3, 4]
    lens = {r: 0 for r in rows}
    while True:
        pre = [lens[r] for r in rows]
        if U.alloc(rows, pre, [p + 3 for p in pre]) is None:
            break
        for r in rows:
            lens[r] += 3
        U.check()
    assert U.o.gap() < 8
    for r in (2, 4, 1, 3):
        idx = [int(x) for x in U.ort[r, :lens[r]]]
        api.swa_unified_free(U.u, torch.tensor(idx, dtype=torch.int64, device="cuda"))
        U.o.free(idx)
        U.rt[r].zero_()
        U.ort[r] = 0
        U.check()
    assert (U.o.low, U.o.high) == (0, 21)
    c = U.u.counters()
    assert (c[api.UCTR_LOW], c[api.UCTR_HIGH], c[api.UCTR_VCOUNT]) == (0, 21, 20)
