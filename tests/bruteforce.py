"""Exact-rational brute force used to pin the oracle (tests only).

Nothing here shares code with the oracle: values are Python Fractions,
binary32 rounding is a textbook round-half-even on an exact rational, and
the e4m3 code is found by a nearest-value search over the finite e4m3
values as torch decodes them (a library routine), with ties going to the
code whose last mantissa bit is 0 and magnitudes at or above 448 saturating
to 448.
"""
from __future__ import annotations

import bisect
import struct
from fractions import Fraction

import torch

# finite non-negative e4m3fn values in code order 0x00..0x7E (torch decode)
_DEC = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
E4M3_VALUES = [Fraction(float(v)) for v in _DEC.tolist()]
assert all(a < b for a, b in zip(E4M3_VALUES, E4M3_VALUES[1:]))
E4M3_MAX = E4M3_VALUES[-1]


def f32_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def f32_from_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def bf16_value(bits: int) -> Fraction:
    return Fraction(f32_from_bits(bits << 16))


def _round_half_even(q: Fraction) -> int:
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def rn_binary32(q: Fraction) -> Fraction:
    """Round an exact rational to the nearest binary32 (ties to even),
    with gradual underflow. Overflow is not needed here and raises."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 23)
    n = _round_half_even(a / quantum)
    r = n * quantum
    if r >= Fraction(2) ** 128:
        raise OverflowError
    return sign * r


def nearest_code(y: Fraction, negative_zero: bool = False) -> int:
    """e4m3fn code of an exact value: nearest finite value, ties to the
    even code, saturating at 448; the sign bit follows the sign of y
    (and of a signed zero via negative_zero)."""
    neg = y < 0 or (y == 0 and negative_zero)
    a = abs(y)
    if a >= E4M3_MAX:
        code = 0x7E
    else:
        i = bisect.bisect_right(E4M3_VALUES, a) - 1     # E4M3_VALUES[i] <= a
        lo, hi = E4M3_VALUES[i], E4M3_VALUES[i + 1]
        if a - lo < hi - a:
            code = i
        elif a - lo > hi - a:
            code = i + 1
        else:
            code = i if i % 2 == 0 else i + 1
    return code | (0x80 if neg else 0)


def block_scale(amax: Fraction) -> Fraction:
    if amax == 0:
        return Fraction(1)
    return rn_binary32(amax / 448)


def element_code(x_bits: int, s: Fraction) -> int:
    x = bf16_value(x_bits)
    y = rn_binary32(x / s)
    return nearest_code(y, negative_zero=bool(x_bits & 0x8000))


def quantize_matrix(bits, rows: int, cols: int):
    """Codes (row-major list) and scale grid (list of Fractions) of a
    rows x cols BF16 matrix given as a flat list of bit patterns."""
    codes = [0] * (rows * cols)
    scales = []
    for bi in range(0, rows, 128):
        for bj in range(0, cols, 128):
            idx = [r * cols + c for r in range(bi, min(bi + 128, rows))
                   for c in range(bj, min(bj + 128, cols))]
            amax = max(abs(bf16_value(bits[i])) for i in idx)
            s = block_scale(amax)
            scales.append(s)
            for i in idx:
                codes[i] = element_code(bits[i], s)
    return codes, scales


def quantize_rows(bits, rows: int, cols: int):
    """Codes (row-major list) and per-row group scales (list of Fractions,
    row-major, ceil(cols/128) per row) of the 1 x 128 activation codec."""
    codes = [0] * (rows * cols)
    scales = []
    for r in range(rows):
        for c0 in range(0, cols, 128):
            idx = [r * cols + c for c in range(c0, min(c0 + 128, cols))]
            amax = max(abs(bf16_value(bits[i])) for i in idx)
            s = block_scale(amax)
            scales.append(s)
            for i in idx:
                codes[i] = element_code(bits[i], s)
    return codes, scales
