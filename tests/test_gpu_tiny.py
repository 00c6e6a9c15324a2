"""End-to-end parity on the Tiny workload: 1 sliding layer (window 16 = 15
prior keys + current) + 1 full layer, Hq=4, Hkv=1, D=64, fp32 KV, page 1,
full pool 512 / SWA pool 128 slots handed out in a seeded permuted order,
two requests decoding at lengths 37 and 200 after a chunked prefill with
eviction before every chunk, then an eviction pass with interval 8.

Allocator outputs, mapping, free lists, req_to_token and stored KV bytes are
compared bit for bit with the oracle after every step; attention outputs to
1e-5 (abs + rel)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from oracle import attention as OT  # noqa: E402
from tests.harness import Pair, assert_close  # noqa: E402

TINY_LAYERS = [(OT.SLIDING, 15, 1), (OT.FULL, 0, 1)]


def _tiny(**kw):
    return Pair(TINY_LAYERS, Hq=4, D=64, dtype="f32", ps=1, size_full=512, size_swa=128,
                perm_free=True, seed=0, **kw)


def _prefill(P, rows, prompt, chunk, evicted):
    lens = np.zeros(len(rows), np.int64)
    while (lens < prompt).any():
        sel = [i for i in range(len(rows)) if lens[i] < prompt[i]]
        ev = evicted[sel].copy()
        P.evict([rows[i] for i in sel], lens[sel], ev, 0)
        evicted[sel] = ev
        new = np.minimum(lens[sel] + chunk, np.asarray(prompt)[sel])
        P.extend([rows[i] for i in sel], lens[sel], new)
        lens[sel] = new
        P.check_state()
    return lens


def test_tiny_end_to_end():
    P = _tiny()
    rows = [1, 2]
    target = np.array([37, 200])
    evicted = np.zeros(2, np.int64)
    lens = _prefill(P, rows, target - 1, 32, evicted)
    # Decode steps: interval-8 eviction, allocate, store, attend.
    for step in range(12):
        P.evict(rows, lens, evicted, 8)
        seq = lens + 1
        P.extend(rows, lens, seq)            # decode = extend by one (checked in alloc test)
        P.check_state()
        res = P.decode_attention(rows, seq)
        for l, (g, o) in res.items():
            assert_close(g, o, 1e-5, f"step {step} layer {l}")
        lens = seq
    assert lens.tolist() == [48, 211]


def test_tiny_alloc_decode_entry_point():
    """The dedicated decode entry point matches the oracle's alloc_decode."""
    from hybrid_sliding_window_gb300 import api
    P = _tiny()
    rows = [1, 2]
    P.extend(rows, [0, 0], [36, 79])     # 115 of the 128 SWA slots
    seq = np.array([37, 80])
    last = [int(P.ort[r, s - 2]) for r, s in zip(rows, seq)]
    out_f = torch.empty(2, dtype=torch.int64, device="cuda")
    out_s = torch.empty(2, dtype=torch.int64, device="cuda")
    api.swa_alloc_decode(P.ctx, torch.tensor(seq, device="cuda"),
                         torch.tensor(last, device="cuda"), seq, out_f, out_s)
    of, osw = P.oa.alloc_decode(seq, last)
    assert out_f.cpu().tolist() == of and out_s.cpu().tolist() == osw
    for r, s, f in zip(rows, seq, of):
        P.ort[r, s - 1] = f
    P.rt[1, 36] = of[0]
    P.rt[2, 79] = of[1]
    P.check_state()
