"""The benchmark's CPU baseline and reference arm on the host (no GPU): the
oracle's whole decode step of one request of the Tiny configuration runs,
and the K+V bytes it reports as attended equal a count made here from the
key sets (a 16-key sliding window and the full prefix, one KV head of 64
float32 values per K and per V row)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from hybrid_sliding_window_gb300.workloads import SPECS  # noqa: E402


def test_oracle_request_step_tiny():
    spec = SPECS["tiny"]
    for b, seq in enumerate(spec.seq_list):
        phases, nbytes, _ = bench.oracle_request_step("tiny", b)
        assert set(phases) == {"evict_alloc", "plan", "store", "attention"}
        assert all(v >= 0 for v in phases.values())
        keys = min(seq, 16) + seq            # sliding layer (window 15 + current) + full layer
        assert nbytes == keys * 1 * 64 * 2 * 4


def test_cpu_model_reports_cores():
    name, n = bench.cpu_model()
    assert isinstance(name, str) and name
    assert n >= 1
