"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times: the whole allocator state against the oracle replaying the same call
trace (bit exact), and sampled attention outputs (all query heads of sampled
requests and layers) against the oracle's brute-force softmax over the
generator's K/V at the attended positions.

Workloads: MiMo-shaped decode (48 layers, B=64, 4K-32K; paged SWA pool and per-request
SWA rings), GPT-OSS-shaped decode
(24 layers, B=128, 1K-16K), Llama4-shaped decode (48 layers, FP8 envelope,
B=16 at 131072), and the MiMo-shaped chunked-prefill extend (B=4, 24576 + 8192)."""
import gc

import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api, synth  # noqa: E402
from hybrid_sliding_window_gb300.workloads import (EXTEND_CHUNK, EXTEND_PREFIX,  # noqa: E402
                                                   EXTEND_SPEC, SPECS, DecodeState, FULL)
from oracle import attention as OT  # noqa: E402
from tests.harness import (OKIND, TOL, assert_close, check_state, oracle_decode,  # noqa: E402
                           replay)


def _free(st):
    del st
    gc.collect()
    torch.cuda.empty_cache()


def _decode_case(name, layers, requests, steps=2, swa_ring=False):
    spec = SPECS[name]
    st = DecodeState(spec, max_steps=steps + 2, trace=True, swa_ring=swa_ring)
    st.prefill()
    st.alloc_decode_buffers()
    inputs = st.make_decode_inputs(steps)
    for s in range(steps):
        st.decode_step(inputs[s])
    torch.cuda.synchronize()
    assert api.swa_last_attn_path(st.ctx) == 1
    oa, ort = replay(st)
    check_state(st, oa, ort)
    last = inputs[-1]
    seq = last["seq_h"]
    reqs = [int(np.argmax(seq)), int(np.argmin(seq))] + list(requests)
    for l in layers:
        g = st.outs[l].float().cpu().numpy()
        q = last["q"][l].float().cpu().numpy()
        for b in reqs:
            o = oracle_decode(st, oa, ort, l, b, seq[b], q[b])
            assert_close(g[b], o, TOL[spec.dtype], f"{name} layer {l} req {b}")
    _free(st)


def test_mimo_decode_full_size():
    _decode_case("mimo", layers=[0, 4, 44, 47], requests=[7])


def test_mimo_decode_full_size_swa_ring():
    """The same workload with per-request SWA rings instead of the paged SWA pool."""
    _decode_case("mimo", layers=[0, 4, 44], requests=[7], swa_ring=True)


def test_gptoss_decode_full_size():
    _decode_case("gptoss", layers=[0, 1, 22, 23], requests=[5])


def test_llama4_decode_full_size():
    spec = SPECS["llama4"]
    st = DecodeState(spec, max_steps=4, trace=True)
    st.prefill()
    st.alloc_decode_buffers()
    inputs = st.make_decode_inputs(2)
    for s in range(2):
        st.decode_step(inputs[s])
    torch.cuda.synchronize()
    oa, ort = replay(st)
    check_state(st, oa, ort)
    last = inputs[-1]
    for l, b in ((0, 3), (3, 0), (46, 11)):
        g = st.outs[l].float().cpu().numpy()
        q = last["q"][l].float().cpu().numpy()
        o = oracle_decode(st, oa, ort, l, b, last["seq_h"][b], q[b])
        assert_close(g[b], o, TOL["e4m3"], f"llama4 layer {l} req {b}")
    _free(st)


def test_extend_full_size_sampled_queries():
    spec = EXTEND_SPEC
    st = DecodeState(spec, max_steps=EXTEND_CHUNK + 64, trace=True, poison_page0=True)
    st.prefill(prompt=np.full(spec.batch, EXTEND_PREFIX, np.int64), final_evict=False)
    meta = st.extend_round(EXTEND_CHUNK)
    torch.cuda.synchronize()
    assert api.swa_last_attn_path(st.ctx) == 2
    # SWA KV below the window was evicted before the chunk (page aligned).
    assert st.evicted.tolist() == [(EXTEND_PREFIX - 127) // 64 * 64] * spec.batch
    oa, ort = replay(st)
    check_state(st, oa, ort)
    rng = np.random.default_rng(0)
    for l in (0, 4, 39):
        kind, w, hkv = spec.layers[l]
        g = meta["out"][l].float().cpu().numpy()
        q = meta["q"][l].float().cpu().numpy()
        for b in range(spec.batch):
            picks = [0, 1, 127, 128, EXTEND_CHUNK - 1] + list(rng.integers(0, EXTEND_CHUNK, 3))
            for i in picks:
                qi = int(meta["indptr"][b] + i)
                p = EXTEND_PREFIX + i
                row = int(st.rows[b])
                J = list(OT.key_positions(OKIND[kind], w, p))
                if kind != FULL:
                    assert all(oa.mapping[int(ort[row, j])] > 0 for j in J)
                K = synth.tokens(spec.seed, synth.STREAM_K, l, [row] * len(J), J, hkv, spec.D)
                V = synth.tokens(spec.seed, synth.STREAM_V, l, [row] * len(J), J, hkv, spec.D)
                o = OT.attend_heads(q[qi].astype(np.float64), K, V, st.sinks_h[l], st.scale)
                assert_close(g[qi], o, TOL["bf16"], f"extend layer {l} req {b} query {i}")
    _free(st)
