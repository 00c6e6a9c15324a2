"""Pins of the oracle's sizing rule against the worked numbers on the pages."""
import json
import os

import pytest

from oracle import attention as A
from oracle import sizing as Z

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_mimo_cell_matches_pages():
    g = _gold("sizing_pages.json")
    F = Z.bytes_per_token_layer(4, 128, 128, 2)   # full layers: 4 KV heads
    S = Z.bytes_per_token_layer(8, 128, 128, 2)   # SWA layers: 8 KV heads
    assert S == 2 * F
    cell = Z.cell_bytes(F, S, g["mimo_full_layers"], g["mimo_swa_layers"], g["r_default"])
    assert cell / F == pytest.approx(g["cell_over_F_r_default"], abs=1e-9)
    swa_part = g["r_default"] * S * g["mimo_swa_layers"]
    assert round(100 * swa_part / cell) == g["swa_share_of_kv_memory_percent_approx"]
    small = Z.cell_bytes(F, S, g["mimo_full_layers"], g["mimo_swa_layers"], g["r_small"])
    assert small / F == pytest.approx(g["cell_over_F_r_small"], abs=1e-9)
    # Same memory, smaller cell: full-pool token capacity grows by cell ratio.
    M = 10 ** 12
    n_big, _ = Z.pool_sizes(M, F, S, 9, 39, g["r_default"], 64, 127)
    n_small, _ = Z.pool_sizes(M, F, S, 9, 39, g["r_small"], 64, 127)
    assert round(n_small / n_big, 1) == g["full_capacity_gain_approx"]


def test_mha_bytes_model_matches_pages():
    g = _gold("pool_bytes_pages.json")
    # kv_heads * (head_dim + v_head_dim) elements = 2 * H * d per token-layer.
    assert Z.bytes_per_token_layer(g["mha_heads"], g["mha_head_dim"], g["mha_head_dim"], 1) \
        == g["mha_elements_per_token_layer"]
    assert g["mla_kv_lora_rank"] + g["mla_rope_dim"] == g["mla_elements_per_token_layer"]


def test_pool_sizes_page_aligned_and_ratio():
    F, S = 2048, 4096
    ps = 64
    for M in (10 ** 9, 7 * 10 ** 10 + 12345, 174 * 10 ** 9):
        nf, ns = Z.pool_sizes(M, F, S, 9, 39, 0.8, ps, 127)
        assert nf % ps == 0 and ns % ps == 0
        assert nf * F * 9 + ns * S * 39 <= M
        # Aligned down from floor(0.8 * floor(M / cell)): at most one page short.
        cell = Z.cell_bytes(F, S, 9, 39, 0.8)
        assert int(M // cell) - nf < ps
        assert 0 <= int(0.8 * int(M // cell)) - ns < ps + 1


def test_pool_sizes_exact_budget():
    F, S, ps = 2048, 4096, 64
    cell = Z.cell_bytes(F, S, 9, 39, 0.5)
    n = 64 * 1000
    nf, ns = Z.pool_sizes(int(cell * n), F, S, 9, 39, 0.5, ps, 127)
    assert nf == n and ns == n // 2


def test_undersized_swa_pool_is_an_error():
    F, S, ps = 2048, 4096, 64
    cell = Z.cell_bytes(F, S, 9, 39, 0.05)
    # floor(M / cell) = 3000 -> N_swa = floor(150) aligned down = 128 <= 127 + 64.
    with pytest.raises(Z.SizingError):
        Z.pool_sizes(int(cell * 3000) + 100, F, S, 9, 39, 0.05, ps, 127)
    # The boundary: N_swa == W + P is an error, one page more is not.
    with pytest.raises(Z.SizingError):
        Z.pool_sizes(int(cell * 2560) + 100, F, S, 9, 39, 0.05, ps, 64)   # N_swa = 128
    nf, ns = Z.pool_sizes(int(cell * 3840) + 100, F, S, 9, 39, 0.05, ps, 64)
    assert (nf, ns) == (3840, 192)


def test_swa_work_ratio_matches_pages():
    g = _gold("swa_ratio_pages.json")
    T, W = g["T"], g["W"]
    # Count attended (query, key) pairs over one sequence of length T.
    full = sum(len(A.key_positions(A.FULL, 0, p)) for p in range(T))
    swa = sum(len(A.key_positions(A.SLIDING, W - 1, p)) for p in range(T))
    ratio = swa / full
    assert ratio < g["ratio_upper_bound"]
    assert ratio == pytest.approx(2 * W / T, rel=0.01)
