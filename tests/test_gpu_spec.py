"""Speculative decode steps on the GPU against the oracle ("SGLang source
teardown (15)", section "how the sizes are set": a request takes alloc_len
slots per step for its draft tree).

Each step: alloc_len slots per request through alloc_extend, their KV
stored, extend attention over the drafted positions; then a verification
keeps a prefix of each request's drafts and returns the pages wholly past it
(the open page stays with the request, as page-granular allocation owns it).
Allocator state bit for bit after every step, attention within the bf16
tolerance; paged SWA pool and per-request rings."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import attention as OT  # noqa: E402
from oracle import sizing as OS  # noqa: E402
from tests.harness import TOL, Pair, assert_close  # noqa: E402

LAYERS = [(OT.SLIDING, 127, 2), (OT.FULL, 0, 2)]


@pytest.mark.parametrize("ring", [0, 400])
def test_speculative_steps(ring):
    ps = 16
    alloc_len, reserve, extra = api.swa_decode_alloc_sizes(OS.SPEC_DRAFT, 3, 4, 8, True, ps)
    assert (alloc_len, reserve, extra) == (128, 256, 271)
    P = Pair(LAYERS, Hq=16, D=128, dtype="bf16", ps=ps, size_full=ps * 256, size_swa=ps * 160,
             seed=11, max_reqs=4, max_ctx=1024, ring_size=ring)
    rows = [1, 2, 3]
    lens = np.array([200, 37, 130], np.int64)
    P.extend(rows, [0, 0, 0], lens)
    evicted = np.zeros(3, np.int64)
    rng = np.random.default_rng(4)
    for step in range(4):
        P.evict(rows, lens, evicted, 0)
        draft_end = lens + alloc_len
        P.extend(rows, lens, draft_end)
        P.check_state()
        for l, (g, o) in P.extend_attention(rows, lens, draft_end).items():
            assert_close(g, o, TOL["bf16"], f"ring {ring} step {step} layer {l}")
        accepted = rng.integers(1, alloc_len + 1, size=3)
        new_len = lens + accepted
        for b, r in enumerate(rows):
            keep_to = -(-int(new_len[b]) // ps) * ps          # the open page stays
            idx = [int(x) for x in P.ort[r, keep_to:draft_end[b]]]
            if idx:
                pages = len(set(i // ps for i in idx))
                swa_pages = 0 if P.ring else len(set(P.oa.mapping[i] // ps for i in idx
                                                     if P.oa.mapping[i] > 0))
                api.swa_free(P.ctx, torch.tensor(idx, dtype=torch.int64, device="cuda"), pages,
                             swa_pages)
                P.oa.free(idx)
            P.rt[r, int(new_len[b]):].zero_()
            P.ort[r, int(new_len[b]):] = 0
        P.check_state()
        lens = new_len
