"""The SWA radix prefix cache driving the device pools ([SWA note], "prefix
cache: tombstones and the window hit rule"), against the oracle allocator
that receives the same releases.

A request is prefilled with eviction before every chunk and handed to the
tree (its slid-out tokens as a tombstone prefix); a second request matches a
shared prefix, locks it, reads it through req_to_token (eviction protected
below the match) and extends from there; SWA eviction then turns unlocked
nodes into tombstones, which moves the usable match end; finally everything
is evicted and every page is back.  Allocator state bit for bit, attention of
the second request within 1e-5."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import attention as OT  # noqa: E402
from tests.harness import Pair, assert_close  # noqa: E402

PS = 4
LAYERS = [(OT.SLIDING, 7, 1), (OT.FULL, 0, 1)]


def _apply(P, T):
    f, live, s = T.apply_releases(P.ctx)
    if len(f):
        P.oa.free([int(x) for x in f])
    if len(s):
        P.oa.free_swa([int(x) for x in s])


def _prefill(P, row, start, n, evicted, protected=0, chunk=16):
    lens = start
    while lens < n:
        ev = np.array([evicted], np.int64)
        P.evict([row], [lens], ev, 0, protected=[protected])
        evicted = int(ev[0])
        new = min(lens + chunk, n)
        P.extend([row], [lens], [new])
        P.check_state()
        res = P.extend_attention([row], [lens], [new])
        for l, (g, o) in res.items():
            assert_close(g, o, 1e-5, f"row {row} [{lens}, {new}) layer {l}")
        lens = new
    return evicted


def test_radix_shares_prefix_and_evicts():
    P = Pair(LAYERS, Hq=2, D=64, dtype="f32", ps=PS, size_full=PS * 128, size_swa=PS * 64,
             seed=3, max_reqs=4, max_ctx=256)
    T = api.RadixSWA(PS, P.lookback)
    full0 = api.swa_available_full(P.ctx)
    rng = np.random.default_rng(0)
    tok_a = rng.integers(1, 50, size=64).tolist()
    ev_a = _prefill(P, 1, 0, 64, 0)
    assert ev_a > 0
    T.insert(tok_a, [int(x) for x in P.ort[1, :64]], ev_a)
    _apply(P, T)
    P.rt[1].zero_()
    P.ort[1] = 0
    P.check_state()
    # request B: shares A's first 48 tokens, then its own
    tok_b = tok_a[:48] + rng.integers(50, 99, size=40).tolist()
    e, slots, node = T.match(tok_b)
    assert e == 48                               # A's tokens past ev_a are live
    span = T.lock(node)
    P.rt[2, :e] = torch.tensor(slots, dtype=torch.int32, device="cuda")
    P.ort[2, :e] = slots
    ev_b = _prefill(P, 2, e, 88, e, protected=e)
    # SWA eviction now: B's lock keeps the W tokens before 48 live
    freed = T.evict(10 ** 6, swa_only=True)
    assert freed > 0
    _apply(P, T)
    P.check_state()
    e2, _, _ = T.match(tok_b)
    assert e2 == 48
    e3, _, _ = T.match(tok_a)                    # A's own tail lost its SWA KV
    assert e3 <= 48
    T.unlock(node, span)
    T.insert(tok_b, [int(x) for x in P.ort[2, :88]], ev_b)
    _apply(P, T)
    P.rt[2].zero_()
    P.ort[2] = 0
    P.check_state()
    T.evict(10 ** 6)
    _apply(P, T)
    P.check_state()
    assert T.sizes() == (0, 0, 0)
    assert api.swa_available_full(P.ctx) == full0
