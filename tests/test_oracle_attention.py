"""Pins of the oracle's attention against library routines and closed forms.

* no sink: the weights are scipy's softmax of the scaled scores;
* a sink is one more logit in the denominator whose value row is zero, so
  the output equals scipy's softmax over ``[scores, sigma]`` with a zero row;
* a single key has the closed form ``v / (1 + exp(sigma - s))``;
* window / chunk masks, GQA head mapping and the score scale agree with
  torch's scaled_dot_product_attention (CPU, float64) given the same mask;
* a window at least as long as the prefix reduces to full causal attention.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import attention as A

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_tiny_window_convention():
    with open(os.path.join(GOLD, "tiny_window.json")) as f:
        g = json.load(f)
    J = A.key_positions(A.SLIDING, g["window_excl"], g["query_position"])
    assert len(J) == g["keys_attended_when_long"]
    assert J[0] == g["first_key"] and J[-1] == g["query_position"]
    assert list(A.key_positions(A.SLIDING, 15, 5)) == list(range(6))


def test_chunked_mask_at_long_context():
    # Llama4-shaped local layer: chunk 8192, query at position 131071.
    J = A.key_positions(A.CHUNKED, 8192, 131071)
    assert J[0] == 122880 and len(J) == 8192
    J = A.key_positions(A.CHUNKED, 8192, 8192)
    assert list(J) == [8192]
    assert A.lookback(A.CHUNKED, 8192) == 8191 and A.lookback(A.SLIDING, 127) == 127


def test_no_sink_is_library_softmax():
    rng = np.random.default_rng(0)
    for n in (1, 2, 7, 100):
        s = rng.normal(size=n) * 3
        np.testing.assert_allclose(A.softmax_with_sink(s, None),
                                   scipy.special.softmax(s), rtol=1e-13)


def test_sink_is_an_extra_logit_with_zero_value():
    rng = np.random.default_rng(1)
    D = 8
    for n in (1, 3, 50):
        q = rng.normal(size=D)
        K = rng.normal(size=(n, D))
        V = rng.normal(size=(n, D))
        sink = rng.normal() * 2
        scale = 0.3
        w = scipy.special.softmax(np.concatenate([scale * K @ q, [sink]]))
        expect = w[:n] @ V + w[n] * np.zeros(D)
        np.testing.assert_allclose(A.attend_one(q, K, V, sink, scale), expect, rtol=1e-12)
        # and without the sink term the result differs (the term matters)
        assert not np.allclose(A.attend_one(q, K, V, None, scale), expect)


def test_single_key_closed_form():
    rng = np.random.default_rng(2)
    q, k, v = rng.normal(size=(3, 16))
    for sink in (-3.0, 0.0, 2.5):
        s = 0.25 * q @ k
        np.testing.assert_allclose(A.attend_one(q, k[None], v[None], sink, 0.25),
                                   v / (1 + np.exp(sink - s)), rtol=1e-12)
    np.testing.assert_allclose(A.attend_one(q, k[None], v[None], None, 0.25), v)


def _sdpa(q, K, V, mask, scale):
    """torch reference for one query: q[Hq, D], K/V[n, Hkv, D], mask[n]."""
    hq, hkv = q.shape[0], K.shape[1]
    g = hq // hkv
    qt = torch.tensor(q)[:, None, :]                         # [Hq, 1, D]
    kt = torch.tensor(K).permute(1, 0, 2).repeat_interleave(g, dim=0)
    vt = torch.tensor(V).permute(1, 0, 2).repeat_interleave(g, dim=0)
    m = torch.tensor(mask)[None, None, :].expand(hq, 1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("kind,window", [(A.FULL, 0), (A.SLIDING, 5), (A.SLIDING, 0),
                                         (A.CHUNKED, 4)])
def test_masks_gqa_scale_against_torch(kind, window):
    rng = np.random.default_rng(3 + kind + window)
    n, hq, hkv, D = 23, 8, 2, 16
    K = rng.normal(size=(n, hkv, D))
    V = rng.normal(size=(n, hkv, D))
    # distinct KV heads so a wrong head mapping cannot pass
    K[:, 1] *= 3.0
    V[:, 1] += 5.0
    scale = 1 / np.sqrt(D)
    for p in (0, 3, 9, 22):
        q = rng.normal(size=(hq, D))
        J = list(A.key_positions(kind, window, p))
        got = A.attend_heads(q, K[J], V[J], None, scale)
        mask = np.zeros(n, dtype=bool)
        mask[J] = True
        want = _sdpa(q, K, V, mask, scale)
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_long_window_reduces_to_causal():
    rng = np.random.default_rng(4)
    n, D = 12, 8
    K = rng.normal(size=(n, 1, D))
    V = rng.normal(size=(n, 1, D))
    q = rng.normal(size=(2, D))
    sinks = rng.normal(size=2)
    for p in range(n):
        a = A.attend_heads(q, K[list(A.key_positions(A.SLIDING, p + 3, p))],
                           V[list(A.key_positions(A.SLIDING, p + 3, p))], sinks, 0.5)
        b = A.attend_heads(q, K[: p + 1], V[: p + 1], sinks, 0.5)
        np.testing.assert_array_equal(a, b)
