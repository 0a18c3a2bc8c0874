"""Pins of the oracle's quantiser and bit-packing against facts that do not come from it."""

import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant

ALL_FP16 = np.arange(0, 1 << 16, dtype=np.uint16).view(np.float16)
POS_FINITE = ALL_FP16[(ALL_FP16 > 0) & np.isfinite(ALL_FP16)]


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_unpack_bijection(bits):
    # every byte value decodes to a code tuple that encodes back to the same byte
    b = np.arange(256, dtype=np.uint8).reshape(256, 1)
    q = quant.unpack(b, bits)
    assert q.shape == (256, 8 // bits)
    assert np.array_equal(quant.pack(q, bits), b)
    # every tuple of storable codes encodes to a byte that decodes back to the tuple
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    tuples = np.array(list(itertools.product(range(lo, hi + 1), repeat=8 // bits)), np.int8)
    assert np.array_equal(quant.unpack(quant.pack(tuples, bits), bits), tuples)
    # and the map is onto all 256 byte values (a bijection)
    assert len(set(quant.pack(tuples, bits)[:, 0].tolist())) == 256


def test_pack_layout_little_endian_hand_worked():
    # INT4: byte j = code[2j] | code[2j+1] << 4, two's complement nibbles.
    # codes (1, -1) -> 0x1 | 0xF<<4 = 0xF1; (7, -7) -> 0x7 | 0x9<<4 = 0x97; (0, -8) -> 0x80
    q4 = np.array([[1, -1, 7, -7, 0, -8, 3, 2]], np.int8)
    assert quant.pack(q4, 4).tolist() == [[0xF1, 0x97, 0x80, 0x23]]
    # INT2: byte j = sum_r code[4j+r] << 2r; (1, -1, 0, 1) -> 1 + 3*4 + 0 + 1*64 = 0x4D
    q2 = np.array([[1, -1, 0, 1, -1, -1, -1, -1]], np.int8)
    assert quant.pack(q2, 2).tolist() == [[0x4D, 0xFF]]


def _nearest_fp16_even(x: Fraction) -> np.float16:
    """Brute force: the finite fp16 nearest to x, ties to the even significand."""
    vals = POS_FINITE
    # bisection on the positive values (sorted, since they are ordered by bit pattern)
    lo, hi = 0, len(vals) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if Fraction(float(vals[mid])) <= x:
            lo = mid
        else:
            hi = mid
    cands = [np.float16(0.0)] + [vals[lo], vals[hi]]
    best = min(cands, key=lambda v: (abs(Fraction(float(v)) - x),
                                     int(np.array(v).view(np.uint16)) & 1))
    return best


@pytest.mark.parametrize("qm", [7, 1])
def test_scale_rounding_fp32_equals_fp64_exhaustive(qm):
    # every positive finite fp16 absmax: fp32 divide + RN16 == fp64 divide + RN16
    a = POS_FINITE
    s32 = (a.astype(np.float32) / np.float32(qm)).astype(np.float16)
    s64 = (a.astype(np.float64) / np.float64(qm)).astype(np.float16)
    assert np.array_equal(s32.view(np.uint16), s64.view(np.uint16))


def test_scale_rounding_matches_exact_rational_nearest():
    rng = np.random.default_rng(7)
    sample = rng.choice(POS_FINITE, size=400, replace=False)
    for a in sample:
        exact = Fraction(float(a)) / 7
        want = _nearest_fp16_even(exact)
        got = (np.float32(a) / np.float32(7)).astype(np.float16)
        assert got.view(np.uint16) == np.float16(want).view(np.uint16), (a, got, want)


def test_code_rounding_fp32_equals_fp64():
    # Over many realistic groups: x / s rounded half-to-even is the same in fp32 and fp64.
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((20000, 32)) * rng.choice([1e-3, 1.0, 30.0], (20000, 1)))
    x16 = x.astype(np.float16)
    a = np.abs(x16.astype(np.float32)).max(-1)
    for qm in (7, 1):
        s = (a / np.float32(qm)).astype(np.float16)
        r32 = np.rint(x16.astype(np.float32) / s.astype(np.float32)[:, None])
        r64 = np.rint(x16.astype(np.float64) / s.astype(np.float64)[:, None])
        assert np.array_equal(r32, r64)


@pytest.mark.parametrize("bits", [2, 4])
def test_dequant_error_bound(bits):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4096, 128)).astype(np.float32)
    x[:, 5] *= 10.0                                        # an outlier channel
    x16 = x.astype(np.float16)
    q, s = quant.quantize(x16, bits)
    qm = quant.qmax(bits)
    assert q.min() >= -qm and q.max() <= qm
    xh = quant.dequantize(q, s)
    err = np.abs(x16.astype(np.float64) - xh).reshape(4096, 4, 32)
    assert np.all(err <= s.astype(np.float64)[..., None] / 2)
    # dequantised values are exactly q*s (checked with rationals on a sample)
    for i, j in [(0, 0), (17, 64), (4095, 127)]:
        assert Fraction(float(xh[i, j])) == int(q[i, j]) * Fraction(float(s[i, j // 32]))


def test_round_half_even_ties():
    # a = 7 -> s = 1 exactly, so x/s = x: half-way values go to the even integer
    g = np.zeros((1, 32), np.float16)
    g[0, :8] = [7.0, 2.5, 3.5, -2.5, 0.5, -0.5, 1.5, -3.5]
    q, s = quant.quantize(g, 4)
    assert float(s[0, 0]) == 1.0
    assert q[0, :8].tolist() == [7, 2, 4, -2, 0, 0, 2, -4]


def test_zero_and_underflow_groups():
    g = np.zeros((2, 64), np.float16)
    g[1, 40] = np.float16(2.0 ** -24)                     # smallest subnormal, alone in group 1
    for bits in (2, 4):
        q, s = quant.quantize(g, bits)
        assert float(s[0, 0]) == 0.0 and float(s[0, 1]) == 0.0 and not q[0].any()
        assert float(s[1, 0]) == 0.0
        assert float(s[1, 1]) == 2.0 ** -24                # underflowed scale floored
        assert q[1, 40] == 1 and np.count_nonzero(q[1]) == 1


def test_int2_is_ternary_sign_of_large_values():
    x = np.array([[3.0, -3.0, 0.4, -0.4, 1.6, -1.6] + [0.0] * 26], np.float16)
    q, s = quant.quantize(x, 2)                            # s = 3, |x| < 1.5 -> 0
    assert float(s[0, 0]) == 3.0
    assert q[0, :6].tolist() == [1, -1, 0, 0, 1, -1]
