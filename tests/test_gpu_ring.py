"""Per-request SWA ring ("SGLang source teardown (15)", section "why sliding
windows can be accounted per request") on the GPU against the oracle.

Chunked prefill (chunks bounded by ring cost - lookback) then decode steps,
with the eviction pass and request frees in between: ring slots, mapping,
full free list, req_to_token and stored KV bytes bit for bit after every
step; decode and extend attention within the dtype tolerance, through the
generic kernel (f32, D = 32), through the tensor-core kernels (bf16,
D = 128, G = 8: keys-as-rows decode and tcgen05 extend) and with E4M3 pools in
the page-major envelope on chunked-local layers (G = 5); every other decode
step stores its new token inside the attention call.  Plus the calls and
configurations ring mode rejects."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import allocator as OA  # noqa: E402
from oracle import attention as OT  # noqa: E402
from tests.harness import TOL, Pair, assert_close  # noqa: E402

CASES = {
    # name: (layers, Hq, D, dtype, ps, ring_size, chunk)
    "f32_generic": ([(OT.SLIDING, 7, 1), (OT.FULL, 0, 1)], 2, 32, "f32", 4, 20, 12),
    "bf16_tensor_core": ([(OT.SLIDING, 127, 2), (OT.FULL, 0, 2)], 16, 128, "bf16", 16, 400, 256),
    # E4M3 pools in the page-major envelope, chunked-local layers, G = 5
    "e4m3_envelope_chunked": ([(OT.CHUNKED, 64, 2), (OT.CHUNKED, 64, 2), (OT.FULL, 0, 2)], 10, 128,
                              "e4m3", 16, 160, 64),
}
EXTRA = {"e4m3_envelope_chunked": dict(layout="envelope", k_scale=0.41, v_scale=1.7)}


def _pair(name):
    layers, Hq, D, dt, ps, ring, _ = CASES[name]
    return Pair(layers, Hq=Hq, D=D, dtype=dt, ps=ps, size_full=ps * 256, size_swa=0, seed=7,
                perm_free=True, max_reqs=6, max_ctx=ps * 64, ring_size=ring,
                **EXTRA.get(name, {}))


@pytest.mark.parametrize("name", list(CASES))
def test_ring_prefill_decode_evict_free(name):
    layers, Hq, D, dt, ps, ring, chunk = CASES[name]
    P = _pair(name)
    assert P.oa.cost - P.lookback >= chunk
    tol = TOL[dt]
    rows = [1, 2, 3]
    target = np.array([3 * chunk + 5, chunk + 1, 2 * chunk - 3])
    lens = np.zeros(3, np.int64)
    evicted = np.zeros(3, np.int64)
    while (lens < target).any():
        sel = [i for i in range(3) if lens[i] < target[i]]
        ev = evicted[sel].copy()
        P.evict([rows[i] for i in sel], lens[sel], ev, 0)
        evicted[sel] = ev
        new = np.minimum(lens[sel] + chunk, target[sel])
        P.extend([rows[i] for i in sel], lens[sel], new)
        P.check_state()
        res = P.extend_attention([rows[i] for i in sel], lens[sel], new)
        for l, (g, o) in res.items():
            assert_close(g, o, tol, f"{name} extend layer {l}")
        lens[sel] = new
    for step in range(6):
        P.evict(rows, lens, evicted, 3)
        seq = lens + 1
        # odd steps: the attention call stores the new token (swa_store_kv_attn_decode)
        fused = step % 2 == 1
        slots = P.extend(rows, lens, seq, store=not fused)
        P.check_state()
        for l, (g, o) in P.decode_attention(rows, seq, new_slots=slots if fused else None).items():
            assert_close(g, o, tol, f"{name} decode step {step} layer {l}")
        lens = seq
    # Request 2 ends: full pages back, its ring slots unmapped.
    r = rows[1]
    idx = [int(x) for x in P.ort[r, :lens[1]]]
    pages = len(set(i // ps for i in idx))
    api.swa_free(P.ctx, torch.tensor(idx, dtype=torch.int64, device="cuda"), pages, 0)
    P.oa.free(idx)
    P.rt[r].zero_()
    P.ort[r] = 0
    P.check_state()
    # Its slot is reused by a new request: the ring takes the new positions.
    P.extend([r], [0], [chunk])
    P.check_state()
    for l, (g, o) in P.extend_attention([r], [0], [chunk]).items():
        assert_close(g, o, tol, f"{name} reuse layer {l}")


def test_ring_rejections():
    P = _pair("f32_generic")
    chunk_max = P.oa.cost - P.lookback
    with pytest.raises(api.SwaError) as e:   # more new tokens than the ring holds
        P.extend([1], [0], [chunk_max + 1], check_alloc=False)
    assert e.value.status == api.SWA_ERR_INVALID
    out = torch.empty(4, dtype=torch.int64, device="cuda")
    with pytest.raises(api.SwaError) as e:   # plain alloc has no request slot
        api.swa_alloc(P.ctx, 4, out, out)
    assert e.value.status == api.SWA_ERR_INVALID
    k = torch.zeros((64 + 4, 1, 32), device="cuda")
    lay = [dict(kind=api.LAYER_SLIDING, window=7, num_kv_heads=1, k=k, v=k)]
    with pytest.raises(api.SwaError) as e:   # size_swa != slots * cost
        api.SwaCtx(lay, 4, 64, 64, 2, 32, api.DTYPE_F32, ring_size=20, ring_slots=3)
    assert e.value.status == api.SWA_ERR_CONFIG
    with pytest.raises(api.SwaError) as e:   # ring shorter than the window
        api.SwaCtx(lay, 4, 64, OA.ring_pool_size(3, 7, 4), 2, 32, api.DTYPE_F32, ring_size=7,
                   ring_slots=3)
    assert e.value.status == api.SWA_ERR_CONFIG
    # The SWA side never runs out; the full pool does.
    assert api.swa_available_swa(P.ctx) == P.oa.size_swa
    assert api.swa_available_size(P.ctx) == api.swa_available_full(P.ctx)
