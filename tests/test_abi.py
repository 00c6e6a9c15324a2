"""The C-ABI library loads without a GPU and exports every symbol the headers
declare; its pure host entry points agree with the oracle."""
import ctypes
import os
import re

import pytest

from hybrid_sliding_window_gb300 import api
from oracle import sizing as Z

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in ("swa.h", "swa_synth.h"):
        txt = open(os.path.join(ROOT, "include", h)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names |= set(re.findall(r"\b(swa_[a-z0-9_]+)\s*\(", txt))
    return names


def test_library_exports_every_declared_symbol():
    if not os.path.exists(api.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    L = ctypes.CDLL(api.LIB_PATH)
    declared = _declared()
    assert len(declared) >= 25
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert declared == set(api.SIGNATURES)
    api.lib()   # binding sets every signature


@pytest.mark.parametrize("M,r,W", [(174 * 10 ** 9, 0.8, 127), (76 * 10 ** 9, 0.05, 8191),
                                   (10 ** 9, 0.5, 127)])
def test_pool_sizes_matches_oracle(M, r, W):
    F = Z.bytes_per_token_layer(4, 128, 128, 2)
    S = Z.bytes_per_token_layer(8, 128, 128, 2)
    want = Z.pool_sizes(M, F, S, 9, 39, r, 64, W)
    assert api.swa_pool_sizes(M, F, S, 9, 39, r, 64, W) == want


def test_pool_sizes_rejects_undersized_swa_pool():
    F, S = 2048, 4096
    cell = Z.cell_bytes(F, S, 9, 39, 0.05)
    with pytest.raises(Z.SizingError):
        Z.pool_sizes(int(cell * 2560) + 100, F, S, 9, 39, 0.05, 64, 64)
    with pytest.raises(api.SwaError) as e:
        api.swa_pool_sizes(int(cell * 2560) + 100, F, S, 9, 39, 0.05, 64, 64)
    assert e.value.status == api.SWA_ERR_CONFIG
