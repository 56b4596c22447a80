"""Pins for the append oracle: bit copy and INT8 quantise-on-append (CPU only)."""

import json
import os

import numpy as np
import pytest

from oracle import append_copy, append_int8, quantize_int8, requantize_int8, bf16_bits_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_copy_round_trip_and_untouched_canaries():
    rng = np.random.default_rng(0)
    NB, Hkv, bs, D = 9, 3, 16, 8
    canary = np.uint16(0xDEAD)
    k = np.full((NB, Hkv, bs, D), canary, dtype=np.uint16)
    v = np.full((NB, Hkv, bs, D), canary, dtype=np.uint16)
    slots = rng.choice(NB * bs, size=40, replace=False).astype(np.int64)
    slots[[3, 17]] = -1
    kn = rng.integers(0, 1 << 16, size=(40, Hkv, D)).astype(np.uint16)
    vn = rng.integers(0, 1 << 16, size=(40, Hkv, D)).astype(np.uint16)
    append_copy(k, v, kn, vn, slots)
    written = np.zeros((NB, bs), dtype=bool)
    for n, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(k[s // bs, :, s % bs], kn[n])
        assert np.array_equal(v[s // bs, :, s % bs], vn[n])
        written[s // bs, s % bs] = True
    assert np.all(k.transpose(0, 2, 1, 3)[~written] == canary)
    assert np.all(v.transpose(0, 2, 1, 3)[~written] == canary)


def _rne_by_definition(y):
    """Nearest integer to the float64 values ``y``, ties to the even one.

    Written with floor and explicit tie logic, independent of ``np.rint``.
    """
    f = np.floor(y)
    d = y - f  # exact for |y| < 2^52
    up = (d > 0.5) | ((d == 0.5) & (np.mod(f, 2.0) == 1.0))
    return f + up


ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
FINITE_BF16 = bf16_bits_to_f32(ALL_BF16)
FINITE_BF16 = FINITE_BF16[np.isfinite(FINITE_BF16)]


@pytest.mark.parametrize("scale", [np.float32(1.0) / np.float32(127.0),
                                   np.float32(3.7) / np.float32(127.0),
                                   np.float32(0.5), np.float32(2.0), np.float32(2.0 ** -20),
                                   np.float32(3.3895314e38) / np.float32(127.0),
                                   np.float32(1e-38)])
def test_quantizer_exhaustive_over_bf16(scale):
    x = FINITE_BF16
    got = quantize_int8(x, scale).astype(np.int64)
    # fp32 quotient via float64 division rounded once to fp32 (innocuous double
    # rounding for division of binary32 operands), then RNE by definition.
    with np.errstate(invalid="ignore", over="ignore"):
        y = np.float32(x.astype(np.float64) / np.float64(scale)).astype(np.float64)
        want = np.clip(_rne_by_definition(y), -127, 127)
    want = np.where(np.isfinite(y), want, np.sign(y) * 127).astype(np.int64)
    assert np.array_equal(got, want)
    # the code is within half a step of the exact ratio wherever it is unclipped
    exact = x.astype(np.float64) / np.float64(scale)
    inside = np.abs(exact) <= 126.5
    assert np.all(np.abs(exact[inside] - got[inside]) <= 0.5 + 1e-6 * np.abs(exact[inside]))


def test_quantizer_zero_scale_gives_zero():
    assert np.all(quantize_int8(FINITE_BF16, np.float32(0.0)) == 0)


def test_requantizer_halving_ties_to_even():
    q = np.array([127, 6, 4, -2, 1, -1, 3, -3], dtype=np.int8)
    got = requantize_int8(q, np.float32(1.0), np.float32(2.0))
    assert got.tolist() == [64, 3, 2, -1, 0, 0, 2, -2]


def _one_tile(D=1):
    return (np.zeros((1, 1, 16, D), np.int8), np.zeros((1, 1, 16, D), np.int8),
            np.zeros((1, 1), np.float32), np.zeros((1, 1), np.float32))


def test_golden_worked_int8_sequence():
    with open(os.path.join(GOLDEN, "int8_append_worked.json")) as f:
        g = json.load(f)
    kc, vc, ks, vs = _one_tile()
    for call in g["calls"]:
        vals = np.array(call["values"], np.float32).reshape(-1, 1, 1)
        append_int8(kc, vc, ks, vs, vals, vals.copy(), np.array(call["slots"], np.int64))
        assert ks[0, 0] == np.float32(call["scale"]) and vs[0, 0] == ks[0, 0]
        assert kc[0, 0, :8, 0].tolist() == call["codes_rows_0_7"]
        assert np.array_equal(vc, kc)


def test_fresh_tile_scale_is_absmax_over_127_and_absmax_codes_127():
    rng = np.random.default_rng(1)
    NB, Hkv, D = 6, 4, 32
    kc = np.zeros((NB, Hkv, 16, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((NB, Hkv), np.float32)
    vs = np.zeros_like(ks)
    slots = np.arange(NB * 16, dtype=np.int64)
    kn = bf16_bits_to_f32((rng.standard_normal((NB * 16, Hkv, D)).astype(np.float32)
                           .view(np.uint32) >> 16).astype(np.uint16))
    vn = 3.0 * kn[::-1].copy()
    append_int8(kc, vc, ks, vs, kn, vn, slots)
    for src, cache, sc in ((kn, kc, ks), (vn, vc, vs)):
        tiles = src.reshape(NB, 16, Hkv, D).transpose(0, 2, 1, 3)
        amax = np.abs(tiles).max(axis=(2, 3))
        assert np.array_equal(sc, (amax / np.float32(127)).astype(np.float32))
        at = np.abs(tiles) == amax[:, :, None, None]
        assert np.all(np.abs(cache[at]) == 127)


def test_scale_monotone_and_final_scale_is_running_absmax():
    rng = np.random.default_rng(2)
    kc, vc, ks, vs = _one_tile(D=8)
    seen = 0.0
    prev = np.float32(0)
    vals_all = []
    for row in range(16):
        x = (rng.standard_normal((1, 1, 8)) * rng.uniform(0.1, 4)).astype(np.float32)
        vals_all.append(x[0, 0])
        append_int8(kc, vc, ks, vs, x, x.copy(), np.array([row], np.int64))
        seen = max(seen, float(np.abs(x).max()))
        assert ks[0, 0] >= prev
        prev = ks[0, 0]
        assert ks[0, 0] == np.float32(np.float32(seen) / np.float32(127))
    # dequantised values stay close: each requantise adds at most half a step
    deq = kc[0, 0].astype(np.float64) * float(ks[0, 0])
    err = np.abs(deq - np.array(vals_all, np.float64))
    assert err.max() <= 16 * 0.5 * float(ks[0, 0]) + 1e-6


def test_reappend_same_values_is_idempotent():
    rng = np.random.default_rng(3)
    NB, Hkv, D = 4, 2, 16
    kc = np.zeros((NB, Hkv, 16, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((NB, Hkv), np.float32)
    vs = np.zeros_like(ks)
    slots = rng.permutation(NB * 16)[:37].astype(np.int64)
    kn = rng.standard_normal((37, Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((37, Hkv, D)).astype(np.float32)
    append_int8(kc, vc, ks, vs, kn, vn, slots)
    snap = (kc.copy(), vc.copy(), ks.copy(), vs.copy())
    append_int8(kc, vc, ks, vs, kn, vn, slots)
    for a, b in zip(snap, (kc, vc, ks, vs)):
        assert np.array_equal(a, b)


def test_zero_rows_then_growth_from_zero_scale():
    kc, vc, ks, vs = _one_tile(D=4)
    z = np.zeros((2, 1, 4), np.float32)
    append_int8(kc, vc, ks, vs, z, z.copy(), np.array([0, 1], np.int64))
    assert ks[0, 0] == 0 and np.all(kc == 0)
    x = np.array([[[1.27, -0.5, 0.0, 0.25]]], np.float32)
    append_int8(kc, vc, ks, vs, x, x.copy(), np.array([2], np.int64))
    assert ks[0, 0] == np.float32(np.float32(1.27) / np.float32(127))
    assert kc[0, 0, 2].tolist() == [127, -50, 0, 25]
    assert np.all(kc[0, 0, :2] == 0)


def test_negative_slots_skip_and_bf16_bits_input():
    kc, vc, ks, vs = _one_tile(D=2)
    bits = np.array([[[0x3F80, 0xC000]], [[0x4000, 0x4000]]], np.uint16)  # (1,-2), (2,2)
    append_int8(kc, vc, ks, vs, bits, bits.copy(), np.array([3, -1], np.int64))
    assert ks[0, 0] == np.float32(np.float32(2.0) / np.float32(127))
    assert kc[0, 0, 3].tolist() == [64, -127]  # 1/(2/127) = 63.5 -> 64 (even)
    assert np.all(np.delete(kc[0, 0], 3, axis=0) == 0)


@pytest.mark.parametrize("mistake", ["half_away", "no_requant", "scale_per_token"])
def test_golden_catches_planted_quantiser_mistakes(mistake):
    """Replay the worked INT8 example through a bugged rule; it must diverge."""
    with open(os.path.join(GOLDEN, "int8_append_worked.json")) as f:
        g = json.load(f)
    codes = np.zeros(16, np.int64)
    s = 0.0
    diverged = False
    for call in g["calls"]:
        vals = np.array(call["values"], np.float64)
        a = np.abs(vals).max()
        sc = a / 127.0
        if mistake == "scale_per_token":
            s = sc
        elif s == 0 or sc > s:
            if s != 0 and mistake != "no_requant":
                codes = np.rint(codes * s / sc).astype(np.int64)
            s = sc
        r = vals / s
        q = np.sign(r) * np.floor(np.abs(r) + 0.5) if mistake == "half_away" else np.rint(r)
        codes[call["slots"]] = np.clip(q, -127, 127)
        if codes[:8].tolist() != call["codes_rows_0_7"] or s != call["scale"]:
            diverged = True
    assert diverged


def test_copy_blocks_round_trip_canaries_and_order():
    from oracle import copy_blocks
    rng = np.random.default_rng(9)
    NB, Hkv, D = 12, 2, 8
    k = rng.integers(0, 1 << 16, size=(NB, Hkv, 16, D)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, size=(NB, Hkv, 16, D)).astype(np.uint16)
    ks = rng.random((NB, Hkv)).astype(np.float32)
    vs = rng.random((NB, Hkv)).astype(np.float32)
    k0, v0, ks0, vs0 = k.copy(), v.copy(), ks.copy(), vs.copy()
    src = np.array([3, 5, 0, 99, 7], np.int32)
    dst = np.array([8, 9, 10, 4, -1], np.int32)    # two pairs out of the pool: skipped
    copy_blocks(k, v, src, dst, ks, vs)
    for s_, d_ in ((3, 8), (5, 9), (0, 10)):
        assert np.array_equal(k[d_], k0[s_]) and np.array_equal(v[d_], v0[s_])
        assert np.array_equal(ks[d_], ks0[s_]) and np.array_equal(vs[d_], vs0[s_])
    untouched = [b for b in range(NB) if b not in (8, 9, 10)]
    assert np.array_equal(k[untouched], k0[untouched])
    assert np.array_equal(ks[untouched], ks0[untouched])
    # pairs apply in order: a chain 1 -> 2 -> 6 carries block 1 to block 6
    k1 = k.copy()
    copy_blocks(k, v, np.array([1, 2]), np.array([2, 6]))
    assert np.array_equal(k[6], k1[1]) and np.array_equal(k[2], k1[1])
