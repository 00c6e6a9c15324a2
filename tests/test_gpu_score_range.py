"""Attention parity on inputs whose scores span a wide range ("SWA in SGLang"
design note, "design": softmax over the window with a per-head sink in the
denominator).

With q, k ~ N(0, 1) the row maxima of neighbouring key blocks differ by a few
units, so code that only runs when a block's maximum jumps far above the
running one is never reached.  These cases reach it:

* queries multiplied by 16 (exact in bf16): every row's scores spread over
  hundreds of log2 units;
* a sawtooth gain on the keys, 1 + (t mod 512) / 16, so that within each
  512-key period every 64-key block beats the previous one by ~14 log2 units;
* (decode) a gain of 4 on the keys of positions 3100-3599, inside one split of
  the longest request, so that split's maximum dominates the others by more
  than 2^8;
* sink logits spread from -200 to +200 across the heads, far below, near and
  far above the scores.

The extend cases prove that the tensor-core kernel's lazy rescale fired: a CPU
model of its block loop (64-key blocks; a block's maximum computed only when
its weights against the reference sum past 2^16, the reference moved when
that maximum exceeds it by more than 8 log2 units) counts rescale events on
the first and on the second block of a 128-key tile over the same inputs, and
the same model with the rescale left out misses the oracle by more than the
tolerance - so a kernel that skipped it would fail here."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import attention as OT  # noqa: E402
from tests.harness import Pair, TOL, assert_close  # noqa: E402

LOG2E = 1.4426950408889634
SINK_SPREAD = np.array([-200.0, -20.0, 0.0, 8.0, 30.0, 60.0, 90.0, 200.0], np.float32)


def sawtooth(pos):
    return 1.0 + (np.asarray(pos) % 512) / 16.0


def bump(pos):
    pos = np.asarray(pos)
    return np.where((pos >= 3100) & (pos < 3600), 4.0, 1.0)


def _spread_sinks(P):
    for l in range(len(P.layers)):
        P.set_sinks(l, np.resize(SINK_SPREAD, P.Hq))


def _build(P, rows, prompt, chunk0=512):
    lens = np.zeros(len(rows), np.int64)
    ev = np.zeros(len(rows), np.int64)
    prompt = np.asarray(prompt, np.int64)
    while (lens < prompt).any():
        sel = [i for i in range(len(rows)) if lens[i] < prompt[i]]
        e = ev[sel].copy()
        P.evict([rows[i] for i in sel], lens[sel], e, 0)
        ev[sel] = e
        new = np.minimum(lens[sel] + chunk0, prompt[sel])
        P.extend([rows[i] for i in sel], lens[sel], new)
        lens[sel] = new
    P.evict(rows, lens, ev, 0)
    return lens


# ---------------------------------------------------------------------------
# CPU model of the extend kernel's block loop (test instrument, not the oracle)
# ---------------------------------------------------------------------------
def lazy_block_softmax(s2, keys, V, sink2, skip_rescale=False):
    """Output of one row by the kernel's loop: 64-key blocks at 64-aligned
    key positions; a block's weights 2^(s - m) are taken against the current
    reference maximum m, and only when there is no reference yet or they sum
    past 2^16 is the block's maximum computed, m moving when that maximum
    exceeds it by more than 8 (log2 units).  Returns (output, rescale events
    on block parity 0, events on parity 1)."""
    m, l = -np.inf, 0.0
    o = np.zeros(V.shape[1])
    ev = [0, 0]
    blocks = keys // 64
    for blk in np.unique(blocks):
        sel = blocks == blk
        if m != -np.inf and (2.0 ** (s2[sel] - m)).sum() <= 65536.0:
            cm = -np.inf      # no maximum pass: the reference stays
        else:
            cm = s2[sel].max()
        if cm > m + 8 or (m == -np.inf and cm != -np.inf):
            if m != -np.inf:
                ev[int(blk) & 1] += 1
                if not skip_rescale:
                    c = 2.0 ** (m - cm)
                    o *= c
                    l *= c
            m = cm
        w = 2.0 ** (s2[sel] - m)
        o += w @ V[sel]
        l += w.sum()
    mf = max(m, sink2) if sink2 is not None else m
    r = 2.0 ** (m - mf)
    den = l * r + (2.0 ** (sink2 - mf) if sink2 is not None else 0.0)
    return o * r / den, ev[0], ev[1]


def _model_rows(P, l, rows, pre, seq, heads):
    """Events and skipped-rescale errors of the model over the chunk's rows."""
    kind, w, hkv = P.layers[l]
    G = P.Hq // hkv
    ev0 = ev1 = 0
    worst = 0.0
    for b, row in enumerate(rows):
        for p in range(int(pre[b]), int(seq[b])):
            J = np.array(list(OT.key_positions(kind, w, p)))
            slots = [int(P.ort[row, j]) for j in J]
            if kind != OT.FULL:
                slots = [P.oa.mapping[s] for s in slots]
            K, V = P.op.read(l, slots, P.k_scale, P.v_scale)
            q = P.q_in(l, [row], [p])[0].astype(np.float64)
            for h in heads:
                s2 = P.scale * LOG2E * (K[:, h // G, :] @ q[h])
                sink2 = float(P.sinks[l][h]) * LOG2E
                good, e0, e1 = lazy_block_softmax(s2, J, V[:, h // G, :], sink2)
                bad, _, _ = lazy_block_softmax(s2, J, V[:, h // G, :], sink2, skip_rescale=True)
                ref = OT.attend_one(q[h], K[:, h // G, :], V[:, h // G, :],
                                    float(P.sinks[l][h]), P.scale)
                assert np.allclose(good, ref, atol=1e-6, rtol=1e-6), (b, p, h)
                ev0 += e0
                ev1 += e1
                worst = max(worst, float((np.abs(bad - ref) / (TOL["bf16"] * (1 + np.abs(ref)))).max()))
    return ev0, ev1, worst


# ---------------------------------------------------------------------------
# extend
# ---------------------------------------------------------------------------
EXTEND_SHAPES = {
    # MiMo-shaped: D = 128, full layer G = 16, page 64
    "mimo": dict(layers=[(OT.SLIDING, 127, 8), (OT.FULL, 0, 4)], D=128, ps=64),
    # GPT-OSS-shaped: D = 64, G = 8, page 16
    "gptoss": dict(layers=[(OT.SLIDING, 127, 8), (OT.FULL, 0, 8)], D=64, ps=16),
}


@pytest.mark.parametrize("shape", list(EXTEND_SHAPES))
@pytest.mark.parametrize("variant", ["q16", "k-sawtooth"])
@pytest.mark.parametrize("path,expect", [pytest.param(-1, 2, id="tcgen05"),
                                         pytest.param(0, 0, id="generic")])
def test_extend_wide_scores(shape, variant, path, expect):
    c = EXTEND_SHAPES[shape]
    ps = c["ps"]
    P = Pair(c["layers"], Hq=64, D=c["D"], dtype="bf16", ps=ps, size_full=ps * (4096 // ps + 40),
             size_swa=ps * (1536 // ps + 40), seed=21, perm_free=True, max_ctx=4096, max_reqs=4)
    api.swa_set_attn_path(P.ctx, path)
    if variant == "q16":
        P.q_gain = 16.0
    else:
        P.k_gain = sawtooth
    _spread_sinks(P)
    rows = [1, 2, 3]
    pre = _build(P, rows, [1500, 700, 0])
    seq = pre + np.array([150, 77, 200])
    P.extend(rows, pre, seq)
    P.check_state()
    res = P.extend_attention(rows, pre, seq)
    assert api.swa_last_attn_path(P.ctx) == expect
    for l, (g, o) in res.items():
        assert np.isfinite(g).all(), f"layer {l}: non-finite output"
        assert_close(g, o, TOL["bf16"], f"{shape} {variant} layer {l}")
    assert api.swa_device_check(P.ctx) == 0
    if path == -1:
        # The inputs drive the rescale on both blocks of a tile, and a loop
        # without it would miss the oracle (full layer, three heads: one per
        # sink regime).
        ev0, ev1, worst = _model_rows(P, 1, rows, pre, seq, heads=(2, 5, 63))
        assert ev0 > 0 and ev1 > 0, (ev0, ev1)
        assert worst > 1.0, worst


# ---------------------------------------------------------------------------
# decode (split-KV with in-launch merge)
# ---------------------------------------------------------------------------
DECODE_CASES = {
    # MiMo full layer: G = 16, heads as the MMA rows
    "bf16-G16": dict(layers=[(OT.FULL, 0, 4)], Hq=64, D=128, dtype="bf16", ps=64),
    # GPT-OSS shape: G = 8, keys as the MMA rows, D = 64
    "bf16-G8-D64": dict(layers=[(OT.SLIDING, 127, 8), (OT.FULL, 0, 8)], Hq=64, D=64,
                        dtype="bf16", ps=16),
    # Llama4 shape: G = 5, E4M3 envelope, a chunked-local layer
    "e4m3-G5-envelope": dict(layers=[(OT.CHUNKED, 2048, 8), (OT.FULL, 0, 8)], Hq=40, D=128,
                             dtype="e4m3", ps=64, layout="envelope"),
}


def _split_dominance(P, l, row, p, h):
    """Maximum of the 1024-key block holding the row's largest score, minus
    the largest maximum of the other blocks (log2 units)."""
    kind, w, hkv = P.layers[l]
    G = P.Hq // hkv
    J = np.array(list(OT.key_positions(kind, w, p)))
    K, _ = P.op.read(l, [int(P.ort[row, j]) for j in J], P.k_scale, P.v_scale)
    q = P.q_in(l, [row], [p])[0].astype(np.float64)
    s2 = P.scale * LOG2E * (K[:, h // G, :] @ q[h])
    maxima = np.array([s2[(J - J[0]) // 1024 == i].max() for i in np.unique((J - J[0]) // 1024)])
    maxima.sort()
    return maxima[-1] - maxima[-2] if len(maxima) > 1 else 0.0


@pytest.mark.parametrize("variant", ["q16", "k-bump"])
@pytest.mark.parametrize("case", list(DECODE_CASES))
@pytest.mark.parametrize("path,expect", [pytest.param(-1, 1, id="mma"),
                                         pytest.param(0, 0, id="generic")])
def test_decode_wide_scores(case, variant, path, expect):
    c = DECODE_CASES[case]
    ps = c["ps"]
    P = Pair(c["layers"], Hq=c["Hq"], D=c["D"], dtype=c["dtype"], ps=ps,
             size_full=ps * (17000 // ps + 40), size_swa=ps * (17000 // ps + 40),
             layout=c.get("layout", "per_layer"), seed=23, perm_free=True, max_ctx=9216,
             max_reqs=4)
    api.swa_set_attn_path(P.ctx, path)
    if variant == "q16":
        P.q_gain = 16.0
    else:
        P.k_gain = bump
    _spread_sinks(P)
    rows = [1, 2, 3]
    lens = _build(P, rows, [9000, 4500, 2100], chunk0=2048)
    seq = lens + 1
    P.extend(rows, lens, seq)
    P.check_state()
    res = P.decode_attention(rows, seq)
    assert api.swa_last_attn_path(P.ctx) == expect
    for l, (g, o) in res.items():
        assert np.isfinite(g).all(), f"layer {l}: non-finite output"
        assert_close(g, o, TOL[c["dtype"]], f"{case} {variant} layer {l}")
    assert api.swa_device_check(P.ctx) == 0
    if variant == "k-bump":
        # The bumped split of the longest request dominates every other split
        # of its full layer by more than 2^8, for every query head.
        full = [l for l, (k, _, _) in enumerate(c["layers"]) if k == OT.FULL][0]
        for h in range(0, c["Hq"], 7):
            assert _split_dominance(P, full, rows[0], int(seq[0]) - 1, h) > 8.0, h
