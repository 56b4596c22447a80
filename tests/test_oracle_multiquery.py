"""Pins for the multi-query (speculative verification / prefill chunk) oracle."""

import json
import os

import numpy as np
from scipy.special import softmax as sp_softmax

from oracle import paged_decode_attention, paged_multiquery_attention
from test_oracle_attention import _random_paged

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cu(ns):
    return np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)


def _dense_causal(q, cu, k, v, t, lens, scale, g, bs=16):
    """Contiguous re-pack + library softmax over an explicit causal mask."""
    out = []
    for b in range(len(lens)):
        n, L = int(cu[b + 1] - cu[b]), int(lens[b])
        if n == 0:
            continue
        nb = -(-L // bs)
        Kc = np.concatenate([k[t[b, j]] for j in range(nb)], axis=1)[:, :L]   # [Hkv, L, D]
        Vc = np.concatenate([v[t[b, j]] for j in range(nb)], axis=1)[:, :L]
        Kq, Vq = np.repeat(Kc, g, axis=0), np.repeat(Vc, g, axis=0)
        Q = q[cu[b]:cu[b + 1]]                                                 # [n, Hq, D]
        S = scale * np.einsum("nhd,hld->nhl", Q, Kq)
        pos = L - n + np.arange(n)
        S = np.where(np.arange(L)[None, None, :] <= pos[:, None, None], S, -np.inf)
        out.append(np.einsum("nhl,hld->nhd", sp_softmax(S, axis=2), Vq))
    return np.concatenate(out)


def test_dense_causal_bruteforce():
    rng = np.random.default_rng(21)
    lens = (5, 16, 17, 40, 73)
    q_, k, v, t, L = _random_paged(rng, lens=lens)
    ns = np.array([3, 1, 17, 5, 9])
    q = rng.standard_normal((int(ns.sum()), 8, 16))
    cu = _cu(ns)
    got = paged_multiquery_attention(q, cu, k, v, t, L, 0.25)
    np.testing.assert_allclose(got, _dense_causal(q, cu, k, v, t, L, 0.25, 4), rtol=0, atol=1e-12)


def test_one_query_per_sequence_is_decode():
    rng = np.random.default_rng(22)
    q, k, v, t, L = _random_paged(rng)
    got = paged_multiquery_attention(q, _cu(np.ones(len(L), int)), k, v, t, L, 0.3)
    np.testing.assert_array_equal(got, paged_decode_attention(q, k, v, t, L, 0.3))


def test_last_query_sees_whole_context_and_causality():
    rng = np.random.default_rng(23)
    q0, k, v, t, L = _random_paged(rng, lens=(40, 73))
    ns = np.array([6, 11])
    cu = _cu(ns)
    q = rng.standard_normal((17, 8, 16))
    a = paged_multiquery_attention(q, cu, k, v, t, L, 0.2)
    last = q[cu[1:] - 1]
    np.testing.assert_array_equal(a[cu[1:] - 1], paged_decode_attention(last, k, v, t, L, 0.2))
    # changing the final token's K/V (position L-1) leaves every earlier query alone
    k2, v2 = k.copy(), v.copy()
    for b in range(2):
        p = int(L[b]) - 1
        k2[t[b, p // 16], :, p % 16] += 5.0
        v2[t[b, p // 16], :, p % 16] -= 3.0
    b_ = paged_multiquery_attention(q, cu, k2, v2, t, L, 0.2)
    keep = np.ones(17, bool)
    keep[cu[1:] - 1] = False
    np.testing.assert_array_equal(a[keep], b_[keep])
    assert not np.allclose(a[~keep], b_[~keep])


def test_golden_worked_multiquery():
    with open(os.path.join(GOLDEN, "multiquery_worked.json")) as f:
        g = json.load(f)
    got = paged_multiquery_attention(np.array(g["q"]), np.array(g["cu_q"]), np.array(g["k_cache"]),
                                     np.array(g["v_cache"]), np.array(g["block_tables"], np.int32),
                                     np.array(g["context_lens"], np.int32), g["softmax_scale"],
                                     block_size=g["block_size"])
    np.testing.assert_allclose(got, np.array(g["expected_out"]), rtol=0, atol=1e-13)
