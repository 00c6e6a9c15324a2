"""Allocator entry points against the oracle, bit for bit: plain alloc,
alloc_extend / alloc_decode, free / free_swa (two-step, double-free safe),
eviction, translate with the -1 sentinel, need_sort staging and merges,
NOMEM leaving every ledger untouched, argument checks, and the device-side
check that flags a window read through an evicted mapping."""
import random

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import allocator as OA  # noqa: E402
from oracle import attention as OT  # noqa: E402
from tests.harness import Pair  # noqa: E402

LAYERS = [(OT.SLIDING, 7, 1), (OT.FULL, 0, 1)]


def _pair(ps, need_sort=False, nf=64, ns=24, seed=1):
    return Pair(LAYERS, Hq=2, D=32, dtype="f32", ps=ps, size_full=ps * nf, size_swa=ps * ns,
                need_sort=need_sort, perm_free=True, seed=seed, max_ctx=ps * nf, max_reqs=8)


def _pages(idx, ps):
    return len(set(int(i) // ps for i in idx))


def _free_gpu(P, idx, swa_only=False):
    """Free through the C-ABI with the page counts a caller knows up front."""
    ps = P.ps
    swa = [P.oa.mapping[int(i)] for i in idx]
    n_swa = len(set(s // ps for s in swa if s > 0))
    t = torch.tensor(idx, dtype=torch.int64, device="cuda")
    if swa_only:
        api.swa_free_swa(P.ctx, t, n_swa)
        P.oa.free_swa(idx)
    else:
        api.swa_free(P.ctx, t, _pages(idx, ps), n_swa)
        P.oa.free(idx)


@pytest.mark.parametrize("ps", [1, 4])
def test_plain_alloc_and_translate(ps):
    P = _pair(ps)
    out_f = torch.empty(ps * 5, dtype=torch.int64, device="cuda")
    out_s = torch.empty(ps * 5, dtype=torch.int64, device="cuda")
    api.swa_alloc(P.ctx, ps * 5, out_f, out_s)
    want = P.oa.alloc(ps * 5)
    assert out_f.cpu().tolist() == want
    assert out_s.cpu().tolist() == P.oa.translate(want)
    q = torch.tensor(want + [-1], dtype=torch.int64, device="cuda")
    res = torch.empty_like(q)
    api.swa_translate(P.ctx, q, res)
    assert res.cpu().tolist() == P.oa.translate(want) + [-1]
    P.check_state()
    with pytest.raises(api.SwaError):   # not page aligned (ps 4) / more than the pools (ps 1)
        api.swa_alloc(P.ctx, ps * 1000 + (1 if ps > 1 else 0), out_f)
    P.check_state()


@pytest.mark.parametrize("ps,need_sort", [(1, False), (4, False), (4, True), (16, True)])
def test_random_sequences_match_oracle(ps, need_sort):
    rnd = random.Random(ps * 7 + need_sort)
    P = _pair(ps, need_sort=need_sort, seed=ps + need_sort)
    lens = {}
    evicted = {}
    for step in range(60):
        op = rnd.random()
        live = sorted(lens)
        if op < 0.5 or not live:
            rows = rnd.sample([r for r in range(1, 8)], rnd.randint(1, 3))
            pre = [lens.get(r, 0) for r in rows]
            seq = [p + rnd.randint(0, 2 * ps + 1) for p in pre]
            need = sum(OA.ceil_div(s, ps) - OA.ceil_div(p, ps) for p, s in zip(pre, seq))
            free_f = P.oa.full.available_size() // ps
            free_s = P.oa.swa.available_size() // ps
            if need > min(free_f, free_s) or max(seq) > P.rt.shape[1]:
                before = (P.ctx.mapping().cpu().clone(), P.ctx.free_list(True), P.ctx.free_list(False))
                if max(seq) <= P.rt.shape[1]:
                    with pytest.raises(api.SwaNoMem):
                        P.extend(rows, pre, seq)
                    # NOMEM: a need_sort merge may have run (as on the pages) - compare sets then
                    assert torch.equal(before[0], P.ctx.mapping().cpu())
                    if not need_sort:
                        assert P.ctx.free_list(True) == before[1]
                        assert P.ctx.free_list(False) == before[2]
                    try:
                        P.oa.alloc_extend(pre, seq, [int(P.ort[r, p - 1]) if p else -1
                                                     for r, p in zip(rows, pre)])
                    except OA.OracleNoMem:
                        pass
                continue
            P.extend(rows, pre, seq)
            for r, s in zip(rows, seq):
                lens[r] = s
                evicted.setdefault(r, 0)
        elif op < 0.7:
            r = rnd.choice(live)
            _free_gpu(P, [int(x) for x in P.ort[r, :lens[r]]])
            del lens[r]
            evicted.pop(r, None)
            P.rt[r].zero_()
            P.ort[r] = 0
        elif op < 0.85:
            r = rnd.choice(live)
            ev = np.array([evicted[r]], np.int64)
            P.evict([r], [lens[r]], ev, rnd.choice([0, 2]))
            evicted[r] = int(ev[0])
        else:
            # free_swa of a page-aligned prefix beyond what eviction freed (then a
            # full free of the request later must not free those pages twice)
            r = rnd.choice(live)
            k = (lens[r] // ps) * ps
            if k > evicted[r]:
                _free_gpu(P, [int(x) for x in P.ort[r, evicted[r]:k]], swa_only=True)
                evicted[r] = k
        P.check_state()
    P.oa.check_no_duplicate_pages()


@pytest.mark.parametrize("need_sort", [False, True])
def test_evict_over_partly_freed_range(need_sort):
    """free_swa of page-aligned parts of two requests, then an eviction pass
    whose ranges cover them ([SWA note], "runtime": free_swa skips tokens
    whose mapping is already 0).  Only the pages still live are released, in
    the oracle's order, no page 0 enters a free list, and the eviction flags
    that its page count differs from the host's (the host counted the whole
    range) until the mirrors are reloaded."""
    P = _pair(4, need_sort=need_sort, nf=64, ns=40)
    P.extend([1, 2], [0, 0], [40, 33])
    _free_gpu(P, [int(x) for x in P.ort[1, 8:20]], swa_only=True)
    _free_gpu(P, [int(x) for x in P.ort[2, 4:8]], swa_only=True)
    P.check_state()
    ev = np.zeros(2, np.int64)
    P.evict([1, 2], [40, 33], ev, 0)          # ranges [0, 32) and [0, 24)
    assert ev.tolist() == [32, 24]
    torch.cuda.synchronize()
    assert api.swa_device_check(P.ctx) == api.SWA_DEVERR_COUNT
    api.swa_sync_counts(P.ctx)
    P.check_state()
    free, staged = P.ctx.free_list(False)
    assert 0 not in free + staged
    assert len(set(free + staged)) == len(free + staged)
    P.oa.check_no_duplicate_pages()


@pytest.mark.parametrize("need_sort", [False, True])
def test_evict_twenty_thousand_slots_in_one_pass(need_sort):
    """One request's out-of-window range of 20 193 tokens at page size 1 is
    released by one eviction call ([SWA note], "runtime":
    free_swa_out_of_window_slots takes the whole range), bit exact against the
    oracle; a second request evicts a short range in the same pass."""
    P = Pair(LAYERS, Hq=2, D=32, dtype="f32", ps=1, size_full=24000, size_swa=22000,
             need_sort=need_sort, perm_free=True, seed=5, max_ctx=20300, max_reqs=3)
    lens = np.zeros(2, np.int64)
    for stop in (6000, 12000, 18000, 20200):
        new = np.array([stop, min(stop // 20, 900)], np.int64)
        P.extend([1, 2], lens, new)
        lens = new
    P.check_state()
    ev = np.zeros(2, np.int64)
    P.evict([1, 2], lens, ev, 0)
    assert ev.tolist() == [20200 - 7, 900 - 7]
    P.check_state()
    P.oa.check_no_duplicate_pages()


def test_free_without_counts_marks_mirror_stale_until_sync():
    P = _pair(4)
    P.extend([1, 2], [0, 0], [9, 13])
    idx = torch.tensor([int(x) for x in P.ort[1, :9]], dtype=torch.int64, device="cuda")
    api.swa_free(P.ctx, idx)                   # counts unknown
    P.oa.free([int(x) for x in P.ort[1, :9]])
    assert api.swa_available_size(P.ctx) == -1
    api.swa_sync_counts(P.ctx)
    assert api.swa_available_size(P.ctx) == P.oa.available_size()


def test_free_count_mismatch_is_flagged():
    P = _pair(4)
    P.extend([1], [0], [9])
    idx = torch.tensor([int(x) for x in P.ort[1, :9]], dtype=torch.int64, device="cuda")
    api.swa_free(P.ctx, idx, 2, 3)               # true counts: 3 and 3
    err = api.swa_device_check(P.ctx)
    assert err & 2                               # SWA_DEVERR_COUNT


def test_window_read_through_evicted_mapping_is_flagged():
    """Freeing SWA slots that are still inside the window (a caller bug) makes
    the plan see mapping 0; the kernel records it instead of trapping."""
    P = _pair(4)
    P.extend([1], [0], [20])
    _free_gpu(P, [int(x) for x in P.ort[1, 12:20]], swa_only=True)
    plan = torch.zeros(api.swa_plan_bytes(P.ctx, 1, 1), dtype=torch.uint8, device="cuda")
    api.swa_plan(P.ctx, P.rt, torch.tensor([1], device="cuda"), None,
                 torch.tensor([20], device="cuda"), plan, 1)
    assert api.swa_device_check(P.ctx) & 1      # SWA_DEVERR_WINDOW_EVICTED
    assert api.swa_device_check(P.ctx) == 0     # the check clears the word


def test_argument_checks():
    P = _pair(4)
    big = np.arange(P.ctx.cfg.max_batch + 1)
    with pytest.raises(api.SwaError) as e:
        api.swa_alloc_extend(P.ctx, torch.zeros(len(big), dtype=torch.int64, device="cuda"),
                             torch.ones(len(big), dtype=torch.int64, device="cuda"), None,
                             np.zeros(len(big), np.int64), np.ones(len(big), np.int64),
                             torch.empty(len(big), dtype=torch.int64, device="cuda"),
                             req_to_token=P.rt, req_idx=torch.zeros(len(big), dtype=torch.int64,
                                                                    device="cuda"))
    assert e.value.status == api.SWA_ERR_INVALID
    with pytest.raises(api.SwaError):
        api.swa_store_kv(P.ctx, 7, torch.zeros((1, 1, 32), device="cuda"),
                         torch.zeros((1, 1, 32), device="cuda"),
                         torch.zeros(1, dtype=torch.int64, device="cuda"))
    with pytest.raises(api.SwaError):
        api.swa_set_attn_path(P.ctx, 5)
    # a decode request must hold at least one token
    with pytest.raises(api.SwaError):
        api.swa_alloc_decode(P.ctx, torch.zeros(1, dtype=torch.int64, device="cuda"), None,
                             np.zeros(1, np.int64), torch.empty(1, dtype=torch.int64, device="cuda"),
                             req_to_token=P.rt, req_idx=torch.ones(1, dtype=torch.int64, device="cuda"))


def test_config_rejections():
    k = torch.zeros((64 + 4, 1, 32), device="cuda")
    base = dict(kind=api.LAYER_SLIDING, window=63, num_kv_heads=1, k=k, v=k)
    with pytest.raises(api.SwaError) as e:       # SWA pool of 64 slots cannot hold W + P
        api.SwaCtx([base], 4, 64, 64, 2, 32, api.DTYPE_F32)
    assert e.value.status == api.SWA_ERR_CONFIG
    env = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    lay = [dict(kind=api.LAYER_FULL, num_kv_heads=1), dict(kind=api.LAYER_SLIDING, window=3,
                                                          num_kv_heads=1)]
    with pytest.raises(api.SwaError) as e:       # envelope without its tail pad
        api.SwaCtx(lay, 4, 16, 16, 2, 32, api.DTYPE_BF16, api.LAYOUT_ENVELOPE,
                   full_envelope=env[:((16 // 4 + 1) * 2 * 4) * 64], swa_envelope=env)
    assert e.value.status == api.SWA_ERR_CONFIG
