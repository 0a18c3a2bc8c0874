"""Arithmetic shortcuts of the CUDA path checked exhaustively on the host with exact rationals.

The quantiser's scale is fp16(fp32(absmax / qmax)) (page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术",
§量化与Bit-Packing: symmetric absmax quantisation). The re-positioning kernel divides with
Markstein's correction step instead of an IEEE division: q0 = a * RN(1/7), e = fma(-q0, 7, a),
q1 = fma(e, RN(1/7), q0). absmax is an fp16 value, so checking every non-negative finite fp16 a
covers every input the kernel can see. Each fp32 operation is emulated exactly (rational
arithmetic, one rounding to nearest-even per operation, as the hardware FMA does).
"""

from fractions import Fraction

import numpy as np


def _rn32(x: Fraction) -> Fraction:
    """Round an exact rational to the nearest fp32 value (ties to even; no overflow here)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    q = x / ulp
    n, rem = divmod(q.numerator, q.denominator)
    rem = Fraction(rem, q.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def test_markstein_division_by_7_is_correctly_rounded_for_every_fp16():
    r = _rn32(Fraction(1, 7))
    assert float(r) == float(np.float32(1.0) / np.float32(7.0))
    fp16 = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    ref = fp16 / np.float32(7.0)  # IEEE fp32 division, round to nearest even
    for a32, want in zip(fp16, ref):
        a = Fraction(float(a32))
        q0 = _rn32(a * r)
        e = _rn32(a - q0 * 7)          # fma(-q0, 7, a): one rounding
        q1 = _rn32(e * r + q0)          # fma(e, r, q0): one rounding
        assert float(q1) == float(want), (float(a32), float(q1), float(want))
