"""Pins of the per-step decode allocation under speculative decoding
("SGLang source teardown (15)", section "how the sizes are set"), and the
C-ABI restatement against the oracle (host arithmetic: no GPU needed)."""
import math

import pytest

from oracle import sizing as S


def test_no_speculation():
    assert S.decode_alloc_len(S.SPEC_NONE, 0, 0, None, 64) == 1
    assert S.decode_reserve(S.SPEC_NONE, 0, 0, None, 64) == 2
    assert S.req_to_token_extra(S.SPEC_NONE, 0, 0, None, 64) == 4


@pytest.mark.parametrize("ps", [2, 4, 16, 64])
@pytest.mark.parametrize("steps", [1, 2, 3, 7, 70])
@pytest.mark.parametrize("topk", [2, 4, 8])
def test_branch_footprint_is_the_worst_page_offset(ps, steps, topk):
    """A branch of `steps` tokens that may start at any slot of a page touches
    at most max over offsets of ceil((offset + steps) / ps) pages; every branch
    gets its own pages."""
    worst = max(math.ceil((o + steps) / ps) for o in range(ps))
    assert S.decode_alloc_len(S.SPEC_DRAFT, steps, topk, 0, ps) == worst * ps * topk
    # the draft-token count wins when it is larger
    big = worst * ps * topk + 5
    assert S.decode_alloc_len(S.SPEC_DRAFT, steps, topk, big, ps) == big


@pytest.mark.parametrize("steps,topk,d", [(3, 4, 8), (5, 1, 6), (4, 2, 3)])
def test_flat_cases(steps, topk, d):
    # page size 1, one branch, or drafts that write no KV: steps x topk or d
    assert S.decode_alloc_len(S.SPEC_DRAFT, steps, topk, d, 1) == max(steps * topk, d)
    assert S.decode_alloc_len(S.SPEC_DRAFT, steps, 1, d, 64) == max(steps, d)
    assert S.decode_alloc_len(S.SPEC_DRAFT, steps, topk, d, 64, has_draft_kv=False) == \
        max(steps * topk, d)
    assert S.req_to_token_extra(S.SPEC_DRAFT, steps, topk, d, 1) == 4 + d


@pytest.mark.parametrize("ps", [1, 16])
def test_uno(ps):
    assert S.decode_alloc_len(S.SPEC_UNO, 0, 0, 8, ps) == 9
    assert S.decode_reserve(S.SPEC_UNO, 0, 0, 8, ps) == 18
    assert S.req_to_token_extra(S.SPEC_UNO, 0, 0, 8, ps) == max(12, 18 + ps - 1)
    with pytest.raises(ValueError):
        S.decode_alloc_len(S.SPEC_UNO, 0, 0, None, ps)


def test_paged_tree_headroom():
    # 3 steps x 4 branches on 64-slot pages: 2 pages per branch -> 512 slots,
    # reserve 1024, headroom 1024 + 63
    assert S.decode_alloc_len(S.SPEC_DRAFT, 3, 4, 8, 64) == 512
    assert S.req_to_token_extra(S.SPEC_DRAFT, 3, 4, 8, 64) == 1087


def test_c_abi_matches_oracle():
    api = pytest.importorskip("hybrid_sliding_window_gb300.api")
    try:
        api.lib()
    except Exception as e:  # library not built here
        pytest.skip(f"libswa not loadable: {e}")
    for algo in (S.SPEC_NONE, S.SPEC_DRAFT, S.SPEC_UNO):
        for ps in (1, 4, 64):
            for steps, topk, d, kv in ((3, 4, 8, True), (1, 1, 0, True), (6, 2, 40, False),
                                       (70, 8, 5, True)):
                got = api.swa_decode_alloc_sizes(algo, steps, topk, d, kv, ps)
                want = (S.decode_alloc_len(algo, steps, topk, d, ps, kv),
                        S.decode_reserve(algo, steps, topk, d, ps, kv),
                        S.req_to_token_extra(algo, steps, topk, d, ps, kv))
                assert got == want, (algo, ps, steps, topk, d, kv)
