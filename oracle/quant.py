"""Symmetric absmax quantisation with bit-packing (oracle).

FADE-zh §量化与Bit-Packing: INT4/INT2 use symmetric quantisation with bit-packing; K stays
INT4 because it is outlier-sensitive, V may go to INT2. FADE-zh §第二层 / §第三层: the
middle tier is 4-bit, optionally 2-bit. The pages fix neither the group, the scale type nor
the packing; the spec fixes them: one fp16 scale per token, per head, per 32-channel group,
codes packed little-endian into uint8.

Readings (no more is stated on the pages):
  * symmetric = mid-tread integer grid, qmax = 2**(bits-1) - 1 (INT4: -7..7, INT2: -1..1);
  * s = fp16(absmax / qmax) rounded to nearest even; absmax = 0 gives s = 0 and all codes 0;
    a positive absmax whose scale underflows to 0 gives s = 2**-24 (smallest fp16 subnormal);
  * q = clamp(round_half_even(x / s), -qmax, qmax);
  * a code is stored as its two's complement truncated to ``bits`` bits; INT4 byte j holds
    channel 2j in bits 0-3 and channel 2j+1 in bits 4-7; INT2 byte j holds channel 4j+r in
    bits 2r..2r+1; channels in natural order;
  * dequantised value = q * s, exact in fp32 and fp64 (a 3-bit integer times an 11-bit
    significand).
Pinned by: exhaustive pack/unpack bijection, exhaustive fp32-vs-fp64 scale rounding over all
positive finite fp16, a brute-force nearest-fp16 search, the |x - q*s| <= s/2 bound,
hand-built round-half-even ties, and zero / underflow groups.
"""

from __future__ import annotations

import numpy as np

GROUP = 32
SUBNORMAL_MIN = np.float16(2.0 ** -24)


def qmax(bits: int) -> int:
    if bits not in (2, 4):
        raise ValueError("bits must be 2 or 4")
    return (1 << (bits - 1)) - 1


def quantize(x16: np.ndarray, bits: int):
    """Quantise fp16 vectors [..., d] (d a multiple of 32).

    Returns (q int8 [..., d], scales fp16 [..., d/32])."""
    x16 = np.asarray(x16, dtype=np.float16)
    d = x16.shape[-1]
    if d % GROUP:
        raise ValueError("head_dim must be a multiple of 32")
    qm = qmax(bits)
    g = x16.reshape(x16.shape[:-1] + (d // GROUP, GROUP)).astype(np.float32)
    a = np.abs(g).max(axis=-1)                               # exact: fp16 values
    s16 = (a / np.float32(qm)).astype(np.float16)             # fp32 IEEE divide, then RN to fp16
    s16 = np.where((a > 0) & (s16 == 0), SUBNORMAL_MIN, s16).astype(np.float16)
    s32 = s16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(g / s32[..., None])                       # fp32 divide, round half to even
    r = np.where(s32[..., None] == 0, np.float32(0), r)
    q = np.clip(r, -qm, qm).astype(np.int8)
    return q.reshape(x16.shape), s16


def pack(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack int8 codes [..., d] into uint8 [..., d*bits/8], little-endian within a byte."""
    per = 8 // bits
    mask = (1 << bits) - 1
    u = (q.astype(np.int16) & mask).astype(np.uint8)
    u = u.reshape(u.shape[:-1] + (u.shape[-1] // per, per))
    out = np.zeros(u.shape[:-1], np.uint8)
    for r in range(per):
        out |= (u[..., r] << np.uint8(bits * r)).astype(np.uint8)
    return out


def unpack(b: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of ``pack``: uint8 [..., n] -> sign-extended int8 codes [..., n*8/bits]."""
    per = 8 // bits
    mask = (1 << bits) - 1
    b = np.asarray(b, np.uint8)
    fields = [((b >> np.uint8(bits * r)) & np.uint8(mask)).astype(np.int16) for r in range(per)]
    u = np.stack(fields, axis=-1).reshape(b.shape[:-1] + (b.shape[-1] * per,))
    u = np.where(u >= (1 << (bits - 1)), u - (1 << bits), u)
    return u.astype(np.int8)


def dequantize(q: np.ndarray, s16: np.ndarray) -> np.ndarray:
    """q [..., d] int8, scales [..., d/32] fp16 -> float64 values q*s (exact)."""
    d = q.shape[-1]
    g = q.reshape(q.shape[:-1] + (d // GROUP, GROUP)).astype(np.float64)
    return (g * s16.astype(np.float64)[..., None]).reshape(q.shape)


def quantize_pack(x16: np.ndarray, bits: int):
    """The codec as one call: fp16 [n, d] -> (packed uint8 [n, d*bits/8], scales fp16)."""
    q, s = quantize(x16, bits)
    return pack(q, bits), s
