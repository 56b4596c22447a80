"""Pins for the float64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: a dense
re-implementation through a library softmax, closed forms, invariants of the
definition, and a hand-worked fixture. Chosen so that a dropped term, a wrong
index (block, row, GQA head) or a transposed operand fails at least one.
"""

import json
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from oracle import decode_kv, merge_states, paged_decode_attention, partial_state

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _random_paged(rng, Hq=8, Hkv=2, D=16, bs=16, lens=(1, 16, 17, 40, 73),
                  extra_blocks=7):
    """Scattered pool with ragged lengths; stale rows filled with huge values."""
    B = len(lens)
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB)
    MB = max(nblk + [1])
    tables = np.full((B, MB), -1, dtype=np.int32)
    c = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[c:c + n]
        c += n
    k = np.full((NB, Hkv, bs, D), 1e30)
    v = np.full((NB, Hkv, bs, D), 1e30)
    for b, L in enumerate(lens):
        for p in range(L):
            blk, r = tables[b, p // bs], p % bs
            k[blk, :, r, :] = rng.standard_normal((Hkv, D))
            v[blk, :, r, :] = rng.standard_normal((Hkv, D))
    q = rng.standard_normal((B, Hq, D))
    return q, k, v, tables, np.array(lens, dtype=np.int32)


def _dense_reference(q, k, v, tables, lens, scale, bs):
    """Re-pack each sequence's blocks contiguously, then dense attention.

    Independent route: concatenate whole logical blocks, truncate to L,
    library softmax over the score matrix of all heads at once.
    """
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        nb = -(-L // bs)
        Kc = np.concatenate([k[tables[b, j]] for j in range(nb)], axis=1)[:, :L]  # [Hkv, L, D]
        Vc = np.concatenate([v[tables[b, j]] for j in range(nb)], axis=1)[:, :L]
        Kq = np.repeat(Kc, g, axis=0)                                              # [Hq, L, D]
        Vq = np.repeat(Vc, g, axis=0)
        S = scale * np.einsum("hd,hld->hl", q[b], Kq)
        P = sp_softmax(S, axis=1)
        out[b] = np.einsum("hl,hld->hd", P, Vq)
    return out


def test_dense_bruteforce_agrees():
    rng = np.random.default_rng(1)
    q, k, v, t, lens = _random_paged(rng)
    got = paged_decode_attention(q, k, v, t, lens, 0.25)
    ref = _dense_reference(q, k, v, t, lens, 0.25, 16)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_block_permutation_invariance():
    rng = np.random.default_rng(2)
    q, k, v, t, lens = _random_paged(rng)
    NB = k.shape[0]
    perm = rng.permutation(NB)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    t2 = np.where(t >= 0, perm[np.maximum(t, 0)], -1).astype(np.int32)
    a = paged_decode_attention(q, k, v, t, lens, 0.3)
    b = paged_decode_attention(q, k2, v2, t2, lens, 0.3)
    np.testing.assert_array_equal(a, b)


def test_uniform_scores_give_mean_of_v():
    rng = np.random.default_rng(3)
    q, k, v, t, lens = _random_paged(rng)
    q[:] = 0.0
    got = paged_decode_attention(q, k, v, t, lens, 1.0)
    g = q.shape[1] // k.shape[1]
    for b, L in enumerate(lens):
        rows = np.stack([v[t[b, p // 16], :, p % 16, :] for p in range(L)])  # [L, Hkv, D]
        mean = rows.mean(axis=0)
        for h in range(q.shape[1]):
            np.testing.assert_allclose(got[b, h], mean[h // g], rtol=0, atol=1e-12)


def test_one_hot_dominant_score_returns_that_row():
    rng = np.random.default_rng(4)
    q, k, v, t, lens = _random_paged(rng, lens=(40, 73, 17))
    Hq, Hkv = q.shape[1], k.shape[1]
    g = Hq // Hkv
    planted = {}
    for b, L in enumerate(lens):
        j = int(rng.integers(0, L))
        planted[b] = j
        for kvh in range(Hkv):
            h = kvh * g  # first query head of the group
            for p in range(L):
                k[t[b, p // 16], kvh, p % 16, :] = 0.0
            k[t[b, j // 16], kvh, j % 16, :] = 100.0 * q[b, h]
    got = paged_decode_attention(q, k, v, t, lens, 1.0)
    for b, L in enumerate(lens):
        j = planted[b]
        for kvh in range(Hkv):
            np.testing.assert_allclose(got[b, kvh * g], v[t[b, j // 16], kvh, j % 16],
                                       rtol=0, atol=1e-12)


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(5)
    q, k, v, t, lens = _random_paged(rng, lens=(1, 1, 1))
    got = paged_decode_attention(q, k, v, t, lens, 0.7)
    g = q.shape[1] // k.shape[1]
    for b in range(3):
        for h in range(q.shape[1]):
            np.testing.assert_array_equal(got[b, h], v[t[b, 0], h // g, 0])


def test_empty_sequence_gives_zeros():
    rng = np.random.default_rng(6)
    q, k, v, t, lens = _random_paged(rng, lens=(0, 5, 0))
    got = paged_decode_attention(q, k, v, t, lens, 0.5)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert np.any(got[1] != 0)


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(7)
    q, k, v, t, lens = _random_paged(rng, Hq=8, Hkv=2)
    g = 4
    k_mha = np.repeat(k, g, axis=1)  # head h of the MHA cache = kv head h // g
    v_mha = np.repeat(v, g, axis=1)
    a = paged_decode_attention(q, k, v, t, lens, 0.2)
    b = paged_decode_attention(q, k_mha, v_mha, t, lens, 0.2)
    np.testing.assert_array_equal(a, b)


def test_gqa_head_mapping_is_contiguous():
    """Only KV head 1 carries signal; query heads 4..7 (not 1,3,5,7) see it."""
    rng = np.random.default_rng(8)
    q, k, v, t, lens = _random_paged(rng, Hq=8, Hkv=2, lens=(20,))
    v[:, 0] = 0.0
    k[:, 0] = 0.0
    got = paged_decode_attention(q, k, v, t, lens, 0.2)
    assert np.all(got[0, :4] == 0)
    assert np.all(np.abs(got[0, 4:]).sum(axis=1) > 0)


def test_split_identity_any_partition():
    rng = np.random.default_rng(9)
    q, k, v, t, lens = _random_paged(rng, lens=(73, 200))
    got = paged_decode_attention(q, k, v, t, lens, 0.25)
    g = q.shape[1] // k.shape[1]
    for b, L in enumerate(lens):
        K = np.stack([k[t[b, p // 16], :, p % 16] for p in range(L)])
        V = np.stack([v[t[b, p // 16], :, p % 16] for p in range(L)])
        for h in range(q.shape[1]):
            s = 0.25 * K[:, h // g] @ q[b, h]
            for trial in range(3):
                cuts = np.sort(rng.choice(np.arange(1, L), size=trial + 2, replace=False))
                edges = [0, *cuts.tolist(), L]
                states = [partial_state(s[a:e], V[a:e, h // g]) for a, e in zip(edges, edges[1:])]
                np.testing.assert_allclose(merge_states(states), got[b, h], rtol=0, atol=1e-12)


def test_merge_of_single_state_is_normalised_sum():
    m, l, o = partial_state(np.array([0.0, np.log(3.0)]), np.array([[4.0], [0.0]]))
    # m is the max score ln 3, so l = exp(-ln 3) + 1 = 4/3 and o = 4 exp(-ln 3) = 4/3
    assert abs(l - 4.0 / 3.0) < 1e-15 and abs(m - np.log(3.0)) < 1e-15
    assert abs(o[0] - 4.0 / 3.0) < 1e-15
    np.testing.assert_allclose(merge_states([(m, l, o)]), [1.0], atol=1e-15)


def test_scale_moves_between_q_and_softmax_scale():
    rng = np.random.default_rng(10)
    q, k, v, t, lens = _random_paged(rng)
    a = paged_decode_attention(q, k, v, t, lens, 0.5)
    b = paged_decode_attention(2.0 * q, k, v, t, lens, 0.25)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_decode_kv_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3FC0, 0x0001, 0x8000, 0x4780], dtype=np.uint16)
    want = [1.0, -2.0, 1.5, 2.0 ** -133, -0.0, 65536.0]
    got = decode_kv(bits)
    assert got.tolist() == want
    assert np.signbit(got[4])
    assert decode_kv(np.array([1.5, -0.25], dtype=np.float16)).tolist() == [1.5, -0.25]
    assert decode_kv(np.array([-127, 5], dtype=np.int8)).tolist() == [-127.0, 5.0]


def test_int8_cache_dequantises_with_block_head_scale():
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, bs = 2, 4, 2, 8, 16
    lens = np.array([20, 9], dtype=np.int32)
    tables = np.array([[3, 1], [0, -1]], dtype=np.int32)
    kq = rng.integers(-127, 128, size=(4, Hkv, bs, D)).astype(np.int8)
    vq = rng.integers(-127, 128, size=(4, Hkv, bs, D)).astype(np.int8)
    ks = rng.uniform(0.001, 0.05, size=(4, Hkv)).astype(np.float32)
    vs = rng.uniform(0.001, 0.05, size=(4, Hkv)).astype(np.float32)
    q = rng.standard_normal((B, Hq, D))
    got = paged_decode_attention(q, kq, vq, tables, lens, 0.3, ks, vs)
    kf = kq.astype(np.float64) * ks.astype(np.float64)[:, :, None, None]
    vf = vq.astype(np.float64) * vs.astype(np.float64)[:, :, None, None]
    ref = _dense_reference(q, kf, vf, tables, lens, 0.3, bs)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_golden_worked_example():
    with open(os.path.join(GOLDEN, "attention_worked.json")) as f:
        g = json.load(f)
    got = paged_decode_attention(np.array(g["q"]), np.array(g["k_cache"]),
                                 np.array(g["v_cache"]),
                                 np.array(g["block_tables"], dtype=np.int32),
                                 np.array(g["context_lens"], dtype=np.int32),
                                 g["softmax_scale"], block_size=g["block_size"])
    np.testing.assert_allclose(got, np.array(g["expected_out"]), rtol=0, atol=1e-13)


def _planted(mistake, q, k_cache, v_cache, block_tables, context_lens, softmax_scale, bs=16):
    """A copy of the oracle's walk with one plausible bug planted."""
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(context_lens[b])
        if L == 0:
            continue
        pos = np.arange(L)
        blk = block_tables[b, pos // bs].astype(np.int64)
        row = (pos // bs) % bs if mistake == "row_from_block" else pos % bs
        K = decode_kv(k_cache[blk, :, row, :])
        V = decode_kv(v_cache[blk, :, row, :])
        for h in range(Hq):
            kvh = h % Hkv if mistake == "mod_head_map" else h // (Hq // Hkv)
            sc = 1.0 if mistake == "no_scale" else softmax_scale
            s = sc * (K[:, kvh] @ q[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w @ (K if mistake == "k_for_v" else V)[:, kvh]) / w.sum()
    return out


@pytest.mark.parametrize("mistake", ["mod_head_map", "row_from_block", "no_scale", "k_for_v"])
def test_pins_catch_planted_mistakes(mistake):
    """The dense pin rejects each planted bug (and accepts the unbugged walk)."""
    rng = np.random.default_rng(12)
    q, k, v, t, lens = _random_paged(rng)
    ref = _dense_reference(q, k, v, t, lens, 0.25, 16)
    np.testing.assert_allclose(_planted(None, q, k, v, t, lens, 0.25), ref, atol=1e-12)
    got = _planted(mistake, q, k, v, t, lens, 0.25)
    assert not np.allclose(got, ref, rtol=0, atol=1e-9)
