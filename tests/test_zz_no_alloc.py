"""swa_attn_decode_noalloc: decode attention for callers that cannot allocate
device memory (their HBM is fully reserved by their own pools, or their host
framework gives them no allocator).  It runs the same kernels with the same
split layout as swa_attn_decode with a caller workspace, so its output must be
identical bit for bit, on two calls in a row (the fixed internal scratch keeps
the previous call's contents: a stale ticket or partial would show), for
layers called right after a layer of another shape (KV-head count, split
count), and for a batch whose scratch is close to the fixed array's size.  A
batch whose scratch would exceed the array is refused.  One step is also
checked against the oracle.

Named so that pytest collects it last."""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from hybrid_sliding_window_gb300.workloads import SPECS, DecodeState, FULL, SLIDING  # noqa: E402
from tests.harness import TOL, assert_close, oracle_decode, replay  # noqa: E402

# MiMo-shaped layers: sliding (8 KV heads) and full (4 KV heads, requests long
# enough for several key splits), alternating, so every call follows a layer
# of another shape.
LAYERS = [(SLIDING, 127, 8), (FULL, 0, 4), (SLIDING, 127, 8), (FULL, 0, 4)]


def _state(trace=False):
    spec = dataclasses.replace(SPECS["mimo"], layers=LAYERS, batch=5,
                               seq_list=(3000, 9500, 200, 12000, 2049), chunk=2048, interval=16)
    st = DecodeState(spec, max_steps=4, trace=trace)
    st.prefill()
    st.alloc_decode_buffers()
    return st


def _noalloc(st, layer, inp, msl=None):
    out = torch.empty_like(st.outs[layer])
    api.swa_attn_decode_noalloc(st.ctx, layer, st.rt, st.rows_d, inp["seq_d"],
                                int(inp["seq_h"].max()) if msl is None else msl, st.plan,
                                inp["q"][layer], st.sinks_d[layer], st.scale, out)
    return out


def test_noalloc_identical_to_workspace_path_twice():
    st = _state(trace=True)
    inputs = st.make_decode_inputs(2)
    for s in range(2):
        inp = inputs[s]
        st.decode_step(inp)            # workspace path: outputs in st.outs
        got = [_noalloc(st, layer, inp) for layer in range(len(LAYERS))]
        torch.cuda.synchronize()
        for layer in range(len(LAYERS)):
            assert torch.equal(got[layer].view(torch.int16), st.outs[layer].view(torch.int16)), \
                f"step {s} layer {layer}"
    assert api.swa_device_check(st.ctx) == 0
    # The last step's no-alloc outputs against the oracle replaying the same calls.
    oa, ort = replay(st)
    inp = inputs[-1]
    for layer in (0, 1):
        g = got[layer].float().cpu().numpy()
        q = inp["q"][layer].float().cpu().numpy()
        for b in range(st.B):
            o = oracle_decode(st, oa, ort, layer, b, inp["seq_h"][b], q[b])
            assert_close(g[b], o, TOL["bf16"], f"oracle layer {layer} req {b}")


def test_noalloc_near_the_scratch_limit():
    """A maximum length whose scratch is just under the array's size is
    accepted and still identical to the workspace path."""
    st = _state()
    inp = st.make_decode_inputs(1)[0]
    st.decode_step(inp)
    cap = api.swa_attn_decode_noalloc_max_bytes()
    lo, hi = int(inp["seq_h"].max()), 1 << 20
    assert api.swa_attn_decode_ws_bytes(st.ctx, 1, st.B, lo) <= cap
    while hi - lo > 1:                  # largest max_seq_len that still fits
        mid = (lo + hi) // 2
        if api.swa_attn_decode_ws_bytes(st.ctx, 1, st.B, mid) <= cap:
            lo = mid
        else:
            hi = mid
    need = api.swa_attn_decode_ws_bytes(st.ctx, 1, st.B, lo)
    assert need > cap * 0.9, (need, cap)
    for layer in (0, 1):
        ws = torch.zeros(api.swa_attn_decode_ws_bytes(st.ctx, layer, st.B, lo), dtype=torch.uint8,
                         device="cuda")
        ref = torch.empty_like(st.outs[layer])
        api.swa_attn_decode(st.ctx, layer, st.rt, st.rows_d, inp["seq_d"], lo, st.plan,
                            inp["q"][layer], st.sinks_d[layer], st.scale, ref, ws)
        got = _noalloc(st, layer, inp, msl=lo)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"layer {layer}"
    assert api.swa_device_check(st.ctx) == 0


def test_noalloc_rejects_oversized_batch():
    st = _state()
    cap = api.swa_attn_decode_noalloc_max_bytes()
    assert cap == 32 << 20
    # A maximum length that needs more split scratch than the fixed array.
    big = 2
    while api.swa_attn_decode_ws_bytes(st.ctx, 1, st.B, big) <= cap:
        big *= 2
    out = torch.empty_like(st.outs[1])
    q = torch.zeros_like(st.outs[1])
    seq = torch.tensor(st.lens + 1, device="cuda")
    with pytest.raises(api.SwaError) as e:
        api.swa_attn_decode_noalloc(st.ctx, 1, st.rt, st.rows_d, seq, big, st.plan, q,
                                    st.sinks_d[1], st.scale, out)
    assert e.value.status == api.SWA_ERR_INVALID
    assert "32 MiB" in str(e.value)
