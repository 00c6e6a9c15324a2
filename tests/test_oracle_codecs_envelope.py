"""Pins of the oracle's element codecs (against torch's conversions) and of the
envelope addressing (against an independent strided view of the buffer), and
of the W-contiguous hit rule (against brute force over tombstone patterns)."""
import itertools

import numpy as np
import pytest
import torch

from oracle import codecs as C
from oracle import envelope as E
from oracle import hitrule as H


# ------------------------------------------------------------- codecs ---
def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = C.e4m3_decode(codes)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and nan.sum() == 2     # 0x7F, 0xFF
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert np.nanmax(ours) == 448.0 and ours[1] == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.normal(size=4000).astype(np.float32) * 30,
        rng.normal(size=2000).astype(np.float32) * 0.01,
        # every midpoint between neighbouring finite codes, both signs
        (lambda v: np.concatenate([(v[1:] + v[:-1]) / 2, -(v[1:] + v[:-1]) / 2]))(
            np.array(sorted(C.e4m3_decode(np.arange(0x7F)))))
    ]).astype(np.float32)
    vals = vals[np.abs(vals) < 448.0]
    ours = C.e4m3_encode(vals)
    ref = torch.tensor(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_saturates_and_scales():
    assert C.e4m3_encode(np.array([1000.0, -1e9, 448.0, 470.0]), 1.0).tolist() == \
        [0x7E, 0xFE, 0x7E, 0x7E]
    assert int(C.e4m3_encode(np.array([np.nan]))[0]) == 0x7F
    # x / scale is taken in float32 before rounding
    assert int(C.e4m3_encode(np.array([3.0]), 2.0)[0]) == int(C.e4m3_encode(np.array([1.5]))[0])
    codes = np.arange(0x7F, dtype=np.uint8)
    assert (C.e4m3_encode(C.e4m3_decode(codes)) == codes).all()


def test_bf16_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(size=5000) * 10, [0.0, -0.0, 1e38, 3.4e38, 1e-40],
                        # exact ties between bf16 neighbours
                        (np.arange(1, 200, dtype=np.float32) * 2 ** -7 + 2 ** -16)]).astype(np.float32)
    ours = C.bf16_encode(x)
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(C.bf16_decode(ours),
                                  torch.tensor(x).to(torch.bfloat16).float().numpy())


# ----------------------------------------------------------- envelope ---
@pytest.mark.parametrize("ps,L", [(1, 1), (4, 3), (16, 2), (64, 4)])
def test_kernel_id_matches_strided_view(ps, L):
    """Dense per-layer views at block offsets address the same bytes as a
    4-D strided [page][block][row] view of the buffer."""
    H, D, item = 2, 4, 1
    row_bytes = H * D * item
    pages = 5
    nbytes = E.envelope_bytes(pages, ps, L, row_bytes) + E.tail_pad_bytes(ps, L, row_bytes)
    n_rows = E.check_envelope(pages, ps, L, D, D, row_bytes, nbytes)
    raw = np.arange(nbytes, dtype=np.int64)
    four_d = np.lib.stride_tricks.as_strided(
        raw, shape=(pages, 2 * L, ps, row_bytes),
        strides=(2 * L * ps * row_bytes * 8, ps * row_bytes * 8, row_bytes * 8, 8))
    seen = set()
    for layer in range(L):
        for is_v in (False, True):
            block = 2 * layer + is_v
            dense = np.lib.stride_tricks.as_strided(
                raw[block * ps * row_bytes:], shape=(n_rows, row_bytes),
                strides=(row_bytes * 8, 8))
            for t in range(pages * ps):
                kid = E.kernel_id(t, ps, L)
                a = dense[kid]
                b = four_d[t // ps, block, t % ps]
                np.testing.assert_array_equal(a, b)
                r = E.row_of(layer, is_v, t, ps, L)
                assert r == E.row_of_strided(layer, is_v, t, ps, L)
                assert r not in seen            # K and V of one id never alias
                seen.add(r)
            # the dense view's last row stays inside the padded buffer
            assert (block * ps + n_rows) * row_bytes <= nbytes


def test_envelope_startup_checks():
    with pytest.raises(E.EnvelopeError):
        E.check_envelope(4, 4, 2, 128, 64, 256, 10 ** 9)                # asymmetric K/V
    rb = 256
    need = E.envelope_bytes(4, 4, 2, rb) + E.tail_pad_bytes(4, 2, rb)
    E.check_envelope(4, 4, 2, 64, 64, rb, need)
    with pytest.raises(E.EnvelopeError):                                 # no tail pad
        E.check_envelope(4, 4, 2, 64, 64, rb, E.envelope_bytes(4, 4, 2, rb))
    # The last view (block 2L-1) ends (2L-1)*ps rows past the envelopes.
    end = (E.envelope_bytes(4, 4, 2, rb) // rb + 3 * 4) * rb
    E.check_envelope(4, 4, 2, 64, 64, rb, end)
    with pytest.raises(E.EnvelopeError):
        E.check_envelope(4, 4, 2, 64, 64, rb, end - 1)
    with pytest.raises(E.EnvelopeError):
        E.check_envelope(2 ** 31 // (2 * 2 * 64) + 1, 64, 2, 64, 64, rb, 2 ** 62)


# ----------------------------------------------------------- hit rule ---
@pytest.mark.parametrize("W", [1, 2, 3, 5])
def test_hit_rule_brute_force(W):
    for n in range(0, 11):
        for bits in itertools.product([False, True], repeat=n):
            ok = H.usable_positions(list(bits), W)
            for e in range(n + 1):
                assert ok[e] == H.usable_brute(list(bits), e, W)
            m = H.match_end(list(bits), n, W)
            assert H.usable_brute(list(bits), m, W)
            assert all(not H.usable_brute(list(bits), e, W) for e in range(m + 1, n + 1))


@pytest.mark.parametrize("ps,L", [(1, 1), (4, 3), (64, 12)])
def test_translate_for_kernel_identity_is_kernel_id(ps, L):
    """With the identity page table the translation is the envelope's
    kernel_id; rows then agree with the independent strided index."""
    pages = 20
    v2p = list(range(pages))
    ts = list(range(pages * ps))
    ids = E.translate_for_kernel(v2p, ts, ps, 2 * L)
    assert ids == [E.kernel_id(t, ps, L) for t in ts]
    for t, i in zip(ts[::7], ids[::7]):
        for l in range(L):
            assert l * 2 * ps + i == E.row_of_strided(l, False, t, ps, L)


def test_translate_for_kernel_tombstone_and_remap():
    ps, m = 4, 6
    v2p = [5, -1, 0, 2]
    ts = [0, 3, 4, 7, 8, 13, 15]
    assert E.translate_for_kernel(v2p, ts, ps, m) == [
        5 * 24 + 0, 5 * 24 + 3,      # page 0 -> physical 5
        0, 0,                        # page 1 is a tombstone: the page-0 sink
        0 * 24 + 0,                  # page 2 -> physical 0
        2 * 24 + 1, 2 * 24 + 3]      # page 3 -> physical 2
