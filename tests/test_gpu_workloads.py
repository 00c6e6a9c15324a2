"""Workload-shaped parity: the GPU decode state (chunked prefill with eviction,
then decode steps) against the oracle replaying the same call trace.

Allocator state (mapping, free lists, req_to_token) is compared bit for bit;
attention outputs of every layer against the oracle's brute-force softmax over
the generator's K/V at the attended positions, after asserting (on the
oracle's own mapping) that every attended SWA key is live."""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from hybrid_sliding_window_gb300.workloads import SPECS, DecodeState, FULL, SLIDING, CHUNKED  # noqa: E402
from tests.harness import TOL, assert_close, check_state, oracle_decode, replay  # noqa: E402

def run_small(spec, steps=3, layers=None, requests=None, path=-1, expect_path=None):
    st = DecodeState(spec, max_steps=steps + 2, trace=True, poison_page0=True)
    api.swa_set_attn_path(st.ctx, path)
    st.prefill()
    st.alloc_decode_buffers()
    inputs = st.make_decode_inputs(steps)
    for s in range(steps):
        st.decode_step(inputs[s])
    oa, ort = replay(st)
    check_state(st, oa, ort)
    last = inputs[-1]
    for l in (layers if layers is not None else range(len(spec.layers))):
        g = st.outs[l].float().cpu().numpy()
        q = last["q"][l].float().cpu().numpy()
        for b in (requests if requests is not None else range(st.B)):
            o = oracle_decode(st, oa, ort, l, b, last["seq_h"][b], q[b])
            assert_close(g[b], o, TOL[spec.dtype], f"{spec.name} layer {l} req {b}")
    if expect_path is not None:
        assert api.swa_last_attn_path(st.ctx) == expect_path
    return st


def small(name, **kw):
    return dataclasses.replace(SPECS[name], **kw)


PATHS = [pytest.param(-1, 1, id="default-cp.async-mma"), pytest.param(0, 0, id="generic")]


@pytest.mark.parametrize("path,expect", PATHS)
def test_mimo_shaped_small(path, expect):
    spec = small("mimo", layers=SPECS["mimo"].layers[:10], batch=4, seq_kind="uniform",
                 seq_lo=100, seq_hi=2500, chunk=256, interval=64)
    run_small(spec, steps=70, path=path, expect_path=expect)  # crosses eviction and page edges


@pytest.mark.parametrize("path,expect", PATHS)
def test_gptoss_shaped_small(path, expect):
    spec = small("gptoss", layers=SPECS["gptoss"].layers[:4], batch=6, seq_lo=200, seq_hi=3000,
                 chunk=512, interval=16)
    run_small(spec, steps=20, path=path, expect_path=expect)


@pytest.mark.parametrize("path,expect", PATHS)
def test_llama4_shaped_small_envelope_fp8(path, expect):
    spec = small("llama4", layers=[(CHUNKED, 256, 8), (CHUNKED, 256, 8), (FULL, 0, 8)] * 2,
                 batch=3, seq_kind="uniform", seq_lo=300, seq_hi=2300, chunk=256, interval=32)
    run_small(spec, steps=40, path=path, expect_path=expect)


@pytest.mark.parametrize("path,expect", PATHS)
def test_split_layers_of_different_shapes_share_workspace(path, expect):
    """Windowed layers long enough to be split, after full layers of another
    shape (more splits, another KV-head count) used the same workspace: the
    split tickets must keep their place whatever the layer's partials size."""
    spec = small("mimo", layers=[(SLIDING, 2999, 8), (FULL, 0, 4), (SLIDING, 2999, 8),
                                 (FULL, 0, 4), (SLIDING, 2999, 8)],
                 batch=3, seq_kind="uniform", seq_lo=4000, seq_hi=9000, chunk=1024, interval=64)
    run_small(spec, steps=3, path=path, expect_path=expect)
    spec = small("llama4", layers=[(CHUNKED, 4096, 8), (FULL, 0, 8), (CHUNKED, 4096, 8)],
                 batch=3, seq_kind="uniform", seq_lo=5000, seq_hi=9000, chunk=1024, interval=64)
    run_small(spec, steps=3, path=path, expect_path=expect)


def test_decode_edge_cases():
    """Length-1 requests (a single key), requests exactly on page and split
    boundaries, and a sliding window longer than the prefix."""
    spec = small("gptoss", layers=[(SLIDING, 127, 8), (FULL, 0, 8)], batch=6,
                 seq_list=(1, 2, 16, 17, 1024, 1025), chunk=64, interval=16)
    st = DecodeState(spec, max_steps=4, trace=True, poison_page0=True)
    st.prefill()
    st.alloc_decode_buffers()
    inputs = st.make_decode_inputs(2)
    for s in range(2):
        st.decode_step(inputs[s])
    oa, ort = replay(st)
    check_state(st, oa, ort)
    for l in range(2):
        g = st.outs[l].float().cpu().numpy()
        q = inputs[-1]["q"][l].float().cpu().numpy()
        for b in range(st.B):
            o = oracle_decode(st, oa, ort, l, b, inputs[-1]["seq_h"][b], q[b])
            assert_close(g[b], o, 2e-2, f"edge layer {l} req {b}")
