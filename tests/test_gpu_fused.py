"""swa_store_kv_attn_decode against swa_store_kv followed by swa_attn_decode
("SGLang source teardown (15)", "who writes into the pages": each layer stores
its new K/V, then attends over it).

Two decode states built from the same seed run the same steps, one with the
fused call and one with the two calls: every pool byte and every attention
output must be identical, on every attention path (the tensor-core kernel
stores the token in its attention launch; the others run the store kernel
first), for bf16 per-layer pools and E4M3 envelope pools, with requests long
enough to be split.  The oracle parity of the fused path itself is covered by
the workload tests, whose decode steps use it.  An out-of-range slot sets the
range error and writes nothing."""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from hybrid_sliding_window_gb300.workloads import FULL, SPECS, DecodeState  # noqa: E402


def _pools(st):
    if st.full_env is not None:
        return [st.full_env, st.swa_env]
    return [t for kv in st.kv for t in kv]


def _pair(spec, steps, path):
    out = []
    for fused in (True, False):
        st = DecodeState(spec, max_steps=steps + 2, poison_page0=True)
        api.swa_set_attn_path(st.ctx, path)
        st.prefill()
        st.alloc_decode_buffers()
        inputs = st.make_decode_inputs(steps)
        outs = []
        for s in range(steps):
            st.decode_step(inputs[s], fused=fused)
            outs.append([o.clone() for o in st.outs])
        torch.cuda.synchronize()
        assert api.swa_device_check(st.ctx) == 0
        out.append((st, outs))
    return out


SPEC_CASES = {
    "mimo-bf16": dataclasses.replace(SPECS["mimo"], layers=SPECS["mimo"].layers[:10], batch=4,
                                     seq_kind="uniform", seq_lo=100, seq_hi=9000, chunk=512,
                                     interval=64),
    "llama4-e4m3-envelope": dataclasses.replace(SPECS["llama4"], layers=SPECS["llama4"].layers[:8],
                                                batch=3, seq_kind="uniform", seq_lo=300,
                                                seq_hi=12000, chunk=1024),
    "gptoss-bf16": dataclasses.replace(SPECS["gptoss"], layers=SPECS["gptoss"].layers[:4], batch=5,
                                       seq_kind="uniform", seq_lo=50, seq_hi=6000, chunk=512),
}


@pytest.mark.parametrize("path", [-1, 0], ids=["mma", "generic"])
@pytest.mark.parametrize("case", list(SPEC_CASES))
def test_fused_equals_two_calls(case, path):
    spec = SPEC_CASES[case]
    (sf, of), (ss, os_) = _pair(spec, 6, path)
    for a, b in zip(_pools(sf), _pools(ss)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    for s, (xs, ys) in enumerate(zip(of, os_)):
        for l, (x, y) in enumerate(zip(xs, ys)):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), (case, path, s, l)


def test_fused_out_of_range_slot_flags_and_skips():
    spec = SPEC_CASES["mimo-bf16"]
    st = DecodeState(spec, max_steps=4)
    st.prefill()
    st.alloc_decode_buffers()
    inp = st.make_decode_inputs(1)[0]
    st.decode_step(inp)
    torch.cuda.synchronize()
    assert api.swa_device_check(st.ctx) == 0
    l = [i for i, (k, _, _) in enumerate(spec.layers) if k == FULL][0]
    k_before = st.kv[l][0].clone()
    bad = torch.full_like(st.out_full, st.size_full + 10 * spec.ps)
    msl = int(inp["seq_h"].max())
    api.swa_store_kv_attn_decode(st.ctx, l, st.rt, st.rows_d, inp["seq_d"], msl, st.plan,
                                 inp["q"][l], inp["k"][l], inp["v"][l], bad, st.out_swa,
                                 st.sinks_d[l], st.scale, st.outs[l], st.ws)
    torch.cuda.synchronize()
    assert api.swa_device_check(st.ctx) & 4                # SWA_DEVERR_RANGE
    assert torch.equal(k_before.view(torch.int16), st.kv[l][0].view(torch.int16))


@pytest.mark.parametrize("dtype,D,G", [("bf16", 128, 16), ("bf16", 64, 4), ("e4m3", 128, 5),
                                       ("f32", 64, 2)])
def test_fused_against_oracle(dtype, D, G):
    """The fused call straight against the oracle (store, then attention over
    the tables), through chunked prefill with eviction: the tensor-core kernel
    for bf16 / E4M3 pools, the generic path (store kernel first) for f32."""
    from oracle import attention as OT
    from tests.harness import Pair, TOL, assert_close
    scales = dict(k_scale=0.37, v_scale=1.9) if dtype == "e4m3" else {}
    P = Pair([(OT.SLIDING, 31, 2), (OT.FULL, 0, 2), (OT.CHUNKED, 64, 2)], Hq=2 * G, D=D,
             dtype=dtype, ps=16, size_full=4096, size_swa=1024, perm_free=True, seed=11, **scales)
    rows = [1, 2, 3, 4]
    lens = np.zeros(4, np.int64)
    ev = np.zeros(4, np.int64)
    for chunk in ([100, 37, 1, 260], [60, 5, 130, 80]):
        P.evict(rows, lens, ev, 0)
        P.extend(rows, lens, lens + np.array(chunk))
        lens = lens + np.array(chunk)
    for _ in range(3):                                   # decode steps
        P.evict(rows, lens, ev, 8)
        slots = P.extend(rows, lens, lens + 1, store=False)
        lens = lens + 1
        P.check_state()
        for l, (g, o) in P.decode_attention(rows, lens, new_slots=slots).items():
            assert_close(g, o, TOL[dtype], f"fused {dtype} layer {l}")
