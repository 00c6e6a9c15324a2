"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times: the whole allocator state against the oracle replaying the same call
trace (bit exact), and attention outputs of every request and every query
head of two layers of each kind against the oracle's brute-force softmax over
the generator's K/V at the attended positions (evaluated on the host's cores).

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
from tests.harness import OKIND, TOL, assert_close, check_state, replay  # noqa: E402
from tests.parallel_oracle import attend_jobs, decode_jobs  # noqa: E402


def _free(st):
    del st
    gc.collect()
    torch.cuda.empty_cache()


def _check_all_requests(st, oa, ort, last, layers):
    """Every request x every query head of `layers` against the oracle."""
    spec = st.spec
    seq = np.asarray(last["seq_h"], np.int64)
    jobs, gpu = [], {}
    for l in layers:
        kind, w, hkv = spec.layers[l]
        # The oracle's queries are drawn on the CPU; the device generator
        # that fed the GPU must have drawn the same values.
        q_cpu = synth.tokens(spec.seed, synth.STREAM_Q, l, st.rows, seq - 1, spec.Hq, spec.D,
                             bf16=spec.dtype != "f32")
        np.testing.assert_array_equal(last["q"][l].float().cpu().numpy(), q_cpu)
        if kind != FULL:     # every attended SWA key is live in the oracle's mapping
            for b, row in enumerate(st.rows):
                J = OT.key_positions(OKIND[kind], w, int(seq[b]) - 1)
                assert all(oa.mapping[int(ort[row, j])] > 0 for j in J), (l, b)
        gpu[l] = st.outs[l].float().cpu().numpy()
        for j in decode_jobs(spec, l, st.rows, seq, q_cpu, st.sinks_h[l], st.scale):
            j["l"] = l
            jobs.append(j)
    for j, o in zip(jobs, attend_jobs(jobs)):
        G = spec.Hq // spec.layers[j["l"]][2]
        g = gpu[j["l"]][j["b"], j["h"] * G:(j["h"] + 1) * G]
        assert_close(g, o[0], TOL[spec.dtype],
                     f"{spec.name} layer {j['l']} req {j['b']} kv head {j['h']}")
    return len(jobs)


def _decode_case(name, layers, steps=2, swa_ring=False):
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
    n = _check_all_requests(st, oa, ort, inputs[-1], layers)
    assert n == st.B * sum(spec.layers[l][2] for l in layers)
    _free(st)


def test_mimo_decode_full_size():
    # sliding layers 0 and 47, full layers 4 and 44: all 64 requests x 64 heads
    _decode_case("mimo", layers=[0, 4, 44, 47])


def test_mimo_decode_full_size_swa_ring():
    """The same workload with per-request SWA rings instead of the paged SWA pool."""
    _decode_case("mimo", layers=[0, 4, 44, 47], swa_ring=True)


def test_gptoss_decode_full_size():
    # sliding layers 0 and 22, full layers 1 and 23: all 128 requests x 64 heads
    _decode_case("gptoss", layers=[0, 1, 22, 23])


def test_llama4_decode_full_size():
    # chunked-local layers 0 and 45, global layers 3 and 47: all 16 requests x 40 heads
    _decode_case("llama4", layers=[0, 3, 45, 47])


def test_extend_full_size_sampled_queries():
    """Two sliding and two full layers; per request the chunk's edge queries
    (first, page and key-tile edges, last) and 24 drawn ones, all query heads."""
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
    jobs, gpu = [], {}
    for l in (0, 4, 39, 44):
        kind, w, hkv = spec.layers[l]
        G = spec.Hq // hkv
        gpu[l] = meta["out"][l]
        for b in range(spec.batch):
            row = int(st.rows[b])
            picks = sorted(set([0, 1, 63, 64, 127, 128, EXTEND_CHUNK - 1]
                               + [int(x) for x in rng.integers(0, EXTEND_CHUNK, 24)]))
            pos = [EXTEND_PREFIX + i for i in picks]
            q = synth.tokens(spec.seed, synth.STREAM_Q, l, [row] * len(pos), pos, spec.Hq, spec.D)
            qi = [int(meta["indptr"][b] + i) for i in picks]
            np.testing.assert_array_equal(meta["q"][l][qi].float().cpu().numpy(), q)
            if kind != FULL:
                for p in pos:
                    assert all(oa.mapping[int(ort[row, j])] > 0
                               for j in OT.key_positions(OKIND[kind], w, p))
            for h in range(hkv):
                jobs.append(dict(seed=spec.seed, layer=l, row=row, kvh=h, D=spec.D, dtype="bf16",
                                 kind=OKIND[kind], window=int(w), pos=pos,
                                 q=q[:, h * G:(h + 1) * G], sinks=st.sinks_h[l][h * G:(h + 1) * G],
                                 scale=st.scale, l=l, h=h, qi=qi, G=G))
    for j, o in zip(jobs, attend_jobs(jobs)):
        G, h = j["G"], j["h"]
        g = gpu[j["l"]][j["qi"], h * G:(h + 1) * G].float().cpu().numpy()
        assert_close(g, o, TOL["bf16"], f"extend layer {j['l']} row {j['row']} kv head {h}")
    _free(st)
