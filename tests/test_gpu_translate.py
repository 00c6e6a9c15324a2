"""Kernel-facing translation through a virtual-to-physical page table ([PR
34602], multi_ended_allocator.py, "translate_kv_loc_for_kernel") on the GPU
against the oracle: random tables with tombstones, every id; ids past the
table read 0 and set the device range flag."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_sliding_window_gb300 import api  # noqa: E402
from oracle import attention as OT  # noqa: E402
from oracle import envelope as E  # noqa: E402
from tests.harness import Pair  # noqa: E402


@pytest.mark.parametrize("ps,mult", [(1, 2), (16, 8), (64, 24)])
def test_translate_for_kernel_matches_oracle(ps, mult):
    rng = np.random.default_rng(ps)
    pages = 300
    v2p = rng.permutation(pages).astype(np.int64) + 1
    v2p[rng.random(pages) < 0.2] = -1
    virt = rng.integers(0, pages * ps, size=5000).astype(np.int64)
    got = api.swa_translate_for_kernel(torch.tensor(v2p, device="cuda"),
                                       torch.tensor(virt, device="cuda"), ps, mult)
    want = E.translate_for_kernel(v2p.tolist(), virt.tolist(), ps, mult)
    assert got.cpu().tolist() == want


def test_translate_for_kernel_range_flag():
    P = Pair([(OT.SLIDING, 3, 1), (OT.FULL, 0, 1)], Hq=1, D=32, dtype="f32", ps=4,
             size_full=64, size_swa=64, oracle=False)
    v2p = torch.tensor([3, -1], dtype=torch.int64, device="cuda")
    virt = torch.tensor([1, 5, 8, -2], dtype=torch.int64, device="cuda")
    out = api.swa_translate_for_kernel(v2p, virt, 4, 2, ctx=P.ctx)
    assert out.cpu().tolist() == [3 * 8 + 1, 0, 0, 0]
    assert api.swa_device_check(P.ctx) & 4        # SWA_DEVERR_RANGE
