"""swa_attn_decode_noalloc: decode attention for callers that cannot allocate
device memory (their HBM is fully reserved by their own pools, or their host
framework gives them no allocator).  It must give the same output as
swa_attn_decode with a caller workspace, on two calls in a row (the fixed
internal scratch keeps the previous call's contents), and refuse a batch whose
scratch would exceed the fixed array.

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
from tests.harness import assert_close  # noqa: E402


def _state():
    # Full layer with requests long enough for several key splits per request.
    spec = dataclasses.replace(SPECS["gptoss"], layers=[(SLIDING, 127, 8), (FULL, 0, 8)],
                               batch=5, seq_list=(3000, 4500, 200, 5000, 2049), chunk=1024,
                               interval=16)
    st = DecodeState(spec, max_steps=4)
    st.prefill()
    st.alloc_decode_buffers()
    return st


def test_noalloc_matches_workspace_path_twice():
    st = _state()
    inputs = st.make_decode_inputs(2)
    for s in range(2):
        inp = inputs[s]
        st.decode_step(inp)            # workspace path: outputs in st.outs
        for layer in range(2):
            ref = st.outs[layer].float().cpu().numpy()
            out = torch.empty_like(st.outs[layer])
            api.swa_attn_decode_noalloc(st.ctx, layer, st.rt, st.rows_d, inp["seq_d"],
                                        st.max_seq_len, st.plan, inp["q"][layer],
                                        st.sinks_d[layer], st.scale, out)
            torch.cuda.synchronize()
            assert_close(out.float().cpu().numpy(), ref, 2e-2, f"step {s} layer {layer}")
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
