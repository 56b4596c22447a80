"""Arithmetic facts the decode kernels rely on, checked on the CPU.

* INT8 codes enter the tensor cores as fp16 values: the byte c + 128 (the code
  XOR 0x80) placed as the low byte under the high byte 0x64 is the fp16 number
  1024 + (c + 128) = 1152 + c, exactly, for every code. The kernels subtract
  the 1152 bias per head afterwards.
* Softmax weights P in [0, 1] enter the P.V products as two 16-bit parts,
  hi = rn(P) and lo = rn(P - hi), with P - hi exact in fp32. For bf16 parts
  hi + lo is within 2^-18 of P (absolute; 2^-16 relative), against 2^-9 for
  a single part; for fp16 parts within 2^-22 |P| (relative, while P - hi is
  in fp16's normal range), against 2^-11.
"""

import numpy as np

from paged_kv_decode_05_gb300.workloads import f32_to_bf16_bits


def _bf16_to_f32(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def test_int8_code_as_biased_fp16_is_exact():
    codes = np.arange(-128, 128, dtype=np.int32)
    low = (codes.astype(np.int8).view(np.uint8) ^ np.uint8(0x80)).astype(np.uint16)
    carrier = (np.uint16(0x6400) | low).view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(carrier, 1152.0 + codes)
    # the same bytes taken from the high half of the word (bytes 2, 3) agree
    word = low.astype(np.uint32) << np.uint32(16)
    hi_half = (((word >> np.uint32(16)) & np.uint32(0xFF)) | np.uint32(0x6400)).astype(np.uint16)
    np.testing.assert_array_equal(hi_half.view(np.float16).astype(np.float64), 1152.0 + codes)


def test_p_split_into_two_16bit_parts():
    rng = np.random.default_rng(0)
    p = np.concatenate([rng.random(200000, dtype=np.float32),
                        np.exp2(-rng.random(20000, dtype=np.float32) * 14).astype(np.float32),
                        np.array([1.0, 0.5, 2.0 ** -14], np.float32)])
    # bf16 parts
    hi = _bf16_to_f32(f32_to_bf16_bits(p))
    r = (p - hi).astype(np.float32)
    assert np.array_equal(r.astype(np.float64), p.astype(np.float64) - hi.astype(np.float64))
    lo = _bf16_to_f32(f32_to_bf16_bits(r))
    err = np.abs((hi.astype(np.float64) + lo) - p)
    assert err.max() <= 2.0 ** -18 and (err / p).max() <= 2.0 ** -16
    one = np.abs(hi.astype(np.float64) - p)
    assert one.max() <= 2.0 ** -9 and one.max() > 2.0 ** -11              # one part is coarser
    # fp16 parts (the INT8 path's operand type), P in fp16's normal range
    hi16 = p.astype(np.float16).astype(np.float32)
    r16 = (p - hi16).astype(np.float32)
    lo16 = r16.astype(np.float16).astype(np.float64)
    normal = np.abs(r16) >= 2.0 ** -14
    rel16 = np.abs((hi16.astype(np.float64) + lo16) - p) / p
    assert rel16[normal].max() <= 2.0 ** -22
    # below fp16's normal range the second part still bounds the absolute error
    assert (np.abs((hi16.astype(np.float64) + lo16) - p)[~normal]).max() <= 2.0 ** -25


def test_int8_single_fp16_weight_error_bound():
    """INT8 caches: the P.V product takes each weight as one fp16 value
    w = rn16(P * s_v) (s_v the block's V scale, P in [0, 1] in fp32) and the
    code carrier's 1152 bias is removed with the sum of those same w, so the
    bias cancels and the output error is that of the rounded weights alone:
    |out - exact| <= 2^-11 max|v| (fp16 rounds normal values within 2^-11
    relative; weights below fp16's normal range are off by at most 2^-25
    absolute). Checked in float64 on short contexts, where single weights are
    largest, and far inside the INT8 bound of 2e-2 for |v| up to ~5."""
    rng = np.random.default_rng(3)
    worst = 0.0
    for _ in range(3000):
        n = int(rng.integers(1, 40))
        codes = rng.integers(-127, 128, n).astype(np.float64)
        sv = np.float32(rng.uniform(0.002, 0.05))
        s = rng.normal(0, 3, n).astype(np.float32)
        p = np.exp2((s - s.max()) * np.float32(1.4426950408889634)).astype(np.float32)
        w = (p * sv).astype(np.float32).astype(np.float16).astype(np.float64)
        l = float(p.astype(np.float64).sum())
        got = (np.sum(w * (1152.0 + codes)) - 1152.0 * w.sum()) / l
        want = float(np.sum(p.astype(np.float64) * codes * np.float64(sv)) / l)
        vmax = float(np.abs(codes).max() * np.float64(sv))
        err = abs(got - want)
        assert err <= 2.0 ** -11 * vmax + 2.0 ** -25 * n * 127 * float(sv) / l + 1e-12
        worst = max(worst, err)
    assert worst < 2e-2 / 8
