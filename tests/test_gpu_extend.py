"""Chunked-prefill (extend) attention parity: the tcgen05 kernel and the generic
kernel against the oracle, MiMo-shaped layers (sliding W=128 with 8 KV heads,
full with 4 KV heads, 64 query heads, D=128, bf16), pages of 16 and 64,
prefixes that end mid-page, chunks that end mid-tile, an empty prefix, and
SWA KV evicted below the window before the chunk (evicted slots poisoned)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import attention as OT  # noqa: E402
from tests.harness import Pair, assert_close  # noqa: E402

LAYERS = [(OT.SLIDING, 127, 8), (OT.FULL, 0, 4)]
GPTOSS_LAYERS = [(OT.SLIDING, 127, 8), (OT.FULL, 0, 8)]      # G = 8, D = 64


def _run(ps, path, prompt, chunk, layers=LAYERS, chunk0=256, D=128, Hq=64, dtype="bf16", **kw):
    P = Pair(layers, Hq=Hq, D=D, dtype=dtype, ps=ps, size_full=ps * (4096 // ps + 40),
             size_swa=ps * (1536 // ps + 40), seed=11, perm_free=True, max_ctx=4096, max_reqs=4,
             **kw)
    api.swa_set_attn_path(P.ctx, path)
    rows = [1, 2, 3]
    lens = np.zeros(3, np.int64)
    ev = np.zeros(3, np.int64)
    prompt = np.asarray(prompt, np.int64)
    while (lens < prompt).any():
        sel = [i for i in range(3) if lens[i] < prompt[i]]
        e = ev[sel].copy()
        P.evict([rows[i] for i in sel], lens[sel], e, 0)
        ev[sel] = e
        new = np.minimum(lens[sel] + chunk0, prompt[sel])
        P.extend([rows[i] for i in sel], lens[sel], new)
        lens[sel] = new
    P.evict(rows, lens, ev, 0)
    seq = lens + np.asarray(chunk, np.int64)
    P.extend(rows, lens, seq)
    P.check_state()
    res = P.extend_attention(rows, lens, seq)
    return P, res


@pytest.mark.parametrize("ps", [16, 64])
@pytest.mark.parametrize("path,expect", [pytest.param(-1, 2, id="tcgen05"),
                                         pytest.param(0, 0, id="generic")])
def test_extend_mimo_shaped(ps, path, expect):
    P, res = _run(ps, path, prompt=[700, 333, 0], chunk=[150, 77, 40])
    assert api.swa_last_attn_path(P.ctx) == expect
    for l, (g, o) in res.items():
        assert_close(g, o, 2e-2, f"ps={ps} layer {l}")
    assert api.swa_device_check(P.ctx) == 0


def test_extend_long_prefix_many_key_tiles():
    """Full layer across many 128-key tiles (prefix 2000, chunk 130)."""
    P, res = _run(64, -1, prompt=[2000, 1290, 5], chunk=[130, 9, 128])
    assert api.swa_last_attn_path(P.ctx) == 2
    for l, (g, o) in res.items():
        assert_close(g, o, 2e-2, f"layer {l}")


@pytest.mark.parametrize("ps", [16, 64])
@pytest.mark.parametrize("path,expect", [pytest.param(-1, 2, id="tcgen05"),
                                         pytest.param(0, 0, id="generic")])
def test_extend_gptoss_shaped_head_dim_64(ps, path, expect):
    """GPT-OSS-shaped layers (D = 64, 8 KV heads, G = 8): the tensor-core
    kernel's 64-column tiles, many key tiles, mid-page prefixes, an empty
    prefix and evicted SWA KV below the window."""
    P, res = _run(ps, path, prompt=[1500, 333, 0], chunk=[150, 77, 40], layers=GPTOSS_LAYERS,
                  D=64)
    assert api.swa_last_attn_path(P.ctx) == expect
    for l, (g, o) in res.items():
        assert_close(g, o, 2e-2, f"D=64 ps={ps} layer {l}")
    assert api.swa_device_check(P.ctx) == 0


CHUNKED_LAYERS = [(OT.CHUNKED, 192, 8), (OT.SLIDING, 63, 8), (OT.FULL, 0, 4)]


@pytest.mark.parametrize("ps", [16, 64])
@pytest.mark.parametrize("path,expect", [pytest.param(-1, 2, id="tcgen05"),
                                         pytest.param(0, 0, id="generic")])
def test_extend_chunked_local_and_short_window(ps, path, expect):
    """Chunked-local attention (keys from the start of the query's 192-token
    chunk: chunk starts fall inside work items and inside 128-key tiles) and a
    64-key sliding window, next to a full layer: the tensor-core kernel's
    windowed instance (per-64-key-chunk masks, chunks outside every row's
    range skipped, whole output tiles by bulk store, ragged ones by the
    warps)."""
    P, res = _run(ps, path, prompt=[700, 333, 0], chunk=[150, 77, 40], layers=CHUNKED_LAYERS)
    assert api.swa_last_attn_path(P.ctx) == expect
    for l, (g, o) in res.items():
        assert_close(g, o, 2e-2, f"chunked ps={ps} layer {l}")
    assert api.swa_device_check(P.ctx) == 0


def test_extend_many_requests():
    """40 requests in one call - the producer's request scan spans two
    32-request batches - with prefixes of 0 to 299 tokens and chunks of 0 to 69
    (three empty ones): the tensor-core kernel against the oracle."""
    rng = np.random.default_rng(5)
    n = 40
    P = Pair(LAYERS, Hq=64, D=128, dtype="bf16", ps=16, size_full=16 * (n * 400 // 16 + 40),
             size_swa=16 * (n * 320 // 16 + 40), seed=13, perm_free=True, max_ctx=512,
             max_reqs=n + 1)
    rows = list(range(1, n + 1))
    prompt = rng.integers(0, 300, n).astype(np.int64)
    chunk = rng.integers(0, 70, n).astype(np.int64)
    chunk[[3, 17, 33]] = 0
    lens = np.zeros(n, np.int64)
    ev = np.zeros(n, np.int64)
    while (lens < prompt).any():
        sel = [i for i in range(n) if lens[i] < prompt[i]]
        e = ev[sel].copy()
        P.evict([rows[i] for i in sel], lens[sel], e, 0)
        ev[sel] = e
        new = np.minimum(lens[sel] + 128, prompt[sel])
        P.extend([rows[i] for i in sel], lens[sel], new)
        lens[sel] = new
    P.evict(rows, lens, ev, 0)
    seq = lens + chunk
    P.extend(rows, lens, seq)
    res = P.extend_attention(rows, lens, seq)
    assert api.swa_last_attn_path(P.ctx) == 2
    for l, (g, o) in res.items():
        assert_close(g, o, 2e-2, f"40 requests layer {l}")
    assert api.swa_device_check(P.ctx) == 0


@pytest.mark.parametrize("Hq,layers", [
    pytest.param(40, [(OT.SLIDING, 127, 8), (OT.CHUNKED, 192, 8), (OT.FULL, 0, 8)], id="G5"),
    pytest.param(24, [(OT.SLIDING, 63, 8), (OT.FULL, 0, 8)], id="G3"),
    pytest.param(8, [(OT.SLIDING, 63, 8), (OT.FULL, 0, 8)], id="G1"),
])
def test_extend_group_sizes_not_dividing_128(Hq, layers):
    """GQA groups whose Q tiles leave rows unused (G = 5: 25 tokens x 5 heads =
    125 rows, G = 3: 126) or hold 128 tokens of one head (G = 1), on the
    tensor-core kernel, against the oracle: Llama4-shaped heads (40 query, 8 KV)
    with bf16 KV, sliding, chunked-local and full layers."""
    P, res = _run(64, -1, prompt=[700, 333, 0], chunk=[150, 77, 40], layers=layers, Hq=Hq)
    assert api.swa_last_attn_path(P.ctx) == 2
    for l, (g, o) in res.items():
        assert_close(g, o, 2e-2, f"Hq={Hq} layer {l}")
    assert api.swa_device_check(P.ctx) == 0


G5_E4M3 = (40, [(OT.CHUNKED, 192, 8), (OT.SLIDING, 127, 8), (OT.FULL, 0, 8)])
G8_E4M3 = (64, LAYERS)


@pytest.mark.parametrize("shape,layout,ps,path,expect", [
    pytest.param(G5_E4M3, "envelope", 64, -1, 2, id="G5-envelope-ps64-tcgen05"),
    pytest.param(G5_E4M3, "per_layer", 16, -1, 2, id="G5-per_layer-ps16-tcgen05"),
    pytest.param(G5_E4M3, "envelope", 64, 0, 0, id="G5-envelope-ps64-generic"),
    pytest.param(G8_E4M3, "per_layer", 64, -1, 2, id="G8-G16-per_layer-ps64-tcgen05"),
    pytest.param(G8_E4M3, "envelope", 16, -1, 2, id="G8-G16-envelope-ps16-tcgen05"),
    pytest.param(G8_E4M3, "per_layer", 64, 0, 0, id="G8-G16-per_layer-ps64-generic"),
])
def test_extend_e4m3(shape, layout, ps, path, expect):
    """E4M3 KV (per-layer pools and the page-major envelope, K and V scales
    0.41 and 1.7): the tensor-core kernel converts K/V to f16 in shared memory
    and runs f16 products; Llama4-shaped heads (G = 5) with chunked-local,
    sliding and full layers, and MiMo-shaped ones, pages of 64 and 16 (a key
    tile over 2 or 8 pages), against the oracle."""
    Hq, layers = shape
    P, res = _run(ps, path, prompt=[700, 333, 0], chunk=[150, 77, 40], layers=layers, Hq=Hq,
                  dtype="e4m3", layout=layout, k_scale=0.41, v_scale=1.7)
    assert api.swa_last_attn_path(P.ctx) == expect
    for l, (g, o) in res.items():
        assert_close(g, o, 2e-2, f"e4m3 {layout} Hq={Hq} layer {l}")
    assert api.swa_device_check(P.ctx) == 0


def test_extend_rejects_misaligned_queries():
    """q or out not 16-byte aligned (the tensor-core kernel moves them by TMA):
    SWA_ERR_INVALID before anything is launched, and the context stays usable."""
    P = Pair(LAYERS, Hq=64, D=128, dtype="bf16", ps=64, size_full=64 * 80, size_swa=64 * 40,
             seed=3, max_ctx=1024, max_reqs=2)
    rows, pre, seq = [1], np.array([0]), np.array([40])
    P.extend(rows, pre, seq)
    d = lambda x: torch.tensor(np.asarray(x, np.int64), device="cuda")
    plan = torch.zeros(api.swa_plan_bytes(P.ctx, 1, 40), dtype=torch.uint8, device="cuda")
    api.swa_plan(P.ctx, P.rt, d(rows), d(pre), d(seq), plan, 40)
    ws = torch.zeros(api.swa_attn_extend_ws_bytes(P.ctx, 1, 40, 40), dtype=torch.uint8,
                     device="cuda")
    buf = torch.zeros(40 * 64 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    good = buf[:40 * 64 * 128].view(40, 64, 128)
    bad = buf[1:1 + 40 * 64 * 128].view(40, 64, 128)      # 2 bytes off
    out = torch.empty_like(good)
    for q, o in ((bad, out), (good, bad)):
        with pytest.raises(api.SwaError) as e:
            api.swa_attn_extend(P.ctx, 1, P.rt, d(rows), d(pre), d(seq), d([0, 40]), 40, 40, 40,
                                plan, q, P.sinks_d[1], P.scale, o, ws)
        assert e.value.status == api.SWA_ERR_INVALID
    api.swa_attn_extend(P.ctx, 1, P.rt, d(rows), d(pre), d(seq), d([0, 40]), 40, 40, 40, plan,
                        good, P.sinks_d[1], P.scale, out, ws)
    torch.cuda.synchronize()
    assert api.swa_device_check(P.ctx) == 0
