"""Decode steps captured in one CUDA graph and replayed once must do exactly
what the same steps issued one by one do: two decode states built from the
same seed run the same steps (crossing an eviction interval), one eagerly and
one through a captured graph; the last step's attention outputs, every KV pool
byte, req_to_token, the mapping and the free lists must be identical, and the
graph-driven state must still match the oracle replaying the call trace."""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from hybrid_sliding_window_gb300.workloads import SPECS, DecodeState  # noqa: E402
from tests.harness import check_state, replay  # noqa: E402

CASES = {
    "mimo-bf16": dataclasses.replace(SPECS["mimo"], layers=SPECS["mimo"].layers[:10], batch=4,
                                     seq_kind="uniform", seq_lo=300, seq_hi=4000, chunk=512,
                                     interval=16),
    "tiny-f32": SPECS["tiny"],
}


def _pools(st):
    if st.full_env is not None:
        return [st.full_env, st.swa_env]
    return [t for kv in st.kv for t in kv]


@pytest.mark.parametrize("case", list(CASES))
def test_graph_replay_equals_eager_steps(case):
    spec = CASES[case]
    steps = 24
    states = []
    for graph in (False, True):
        st = DecodeState(spec, max_steps=steps + 4, trace=graph)
        st.prefill()
        st.alloc_decode_buffers()
        inputs = st.make_decode_inputs(steps)
        ev0 = st.evicted.copy()
        torch.cuda.synchronize()
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for inp in inputs:
                    st.decode_step(inp)
            g.replay()
        else:
            for inp in inputs:
                st.decode_step(inp)
        torch.cuda.synchronize()
        assert api.swa_device_check(st.ctx) == 0
        assert (st.evicted != ev0).any(), "the steps should cross an eviction interval"
        states.append(st)
    eager, graphed = states
    for a, b in zip(eager.outs, graphed.outs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    for a, b in zip(_pools(eager), _pools(graphed)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert torch.equal(eager.rt, graphed.rt)
    assert torch.equal(eager.ctx.mapping(), graphed.ctx.mapping())
    for full in (True, False):
        assert eager.ctx.free_list(full) == graphed.ctx.free_list(full)
    np.testing.assert_array_equal(eager.evicted_d.cpu().numpy(), graphed.evicted_d.cpu().numpy())
    oa, ort = replay(graphed)
    check_state(graphed, oa, ort)
