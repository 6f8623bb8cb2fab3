"""The oracle's e4m3 encoder on every one of the 2^32 fp32 bit patterns.

Reference: a nearest-code search over the format's 127 finite non-negative
magnitudes, each decoded from the definition (code c: exponent field c >> 3,
mantissa c & 7; subnormal m 2^-9 for a zero exponent field, else
(1 + m / 8) 2^(e - 7)), picking the nearer neighbour of |y| and, on an exact
tie, the code with an even mantissa; |y| >= 448 (including infinity)
saturates to 0x7E; the sign bit is y's. This search runs on every pattern
with 2^-11 <= |y| < 512 (20 binades, where codes other than 0 and 0x7E
occur); below that the code must be the signed zero, above it the signed
saturation, and NaN patterns must give a NaN code. Negative patterns must
give their positive twin's code with the sign bit set."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from gpu_helpers import ncores

SUB = 1 << 24


def _magnitudes():
    c = np.arange(127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e - 7))


def _nearest_codes(bits):
    """Code of each non-negative fp32 pattern by nearest-code search."""
    v = _magnitudes()
    a = bits.view(np.float32).astype(np.float64)
    hi = np.searchsorted(v, a, side="left").clip(1, 126)
    lo = hi - 1
    d_lo, d_hi = a - v[lo], v[hi] - a
    code = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(a >= 448.0, 126, code)
    return code.astype(np.uint8)


def _encode(oracle_mod, first, n, ex):
    return np.concatenate(list(ex.map(lambda k: oracle_mod.e4m3_encode_bits_range(first + k, min(SUB, n - k)),
                                      range(0, n, SUB))))


def test_every_fp32_pattern(oracle_mod):
    lo_bits = np.float32(2.0 ** -11).view(np.uint32)      # 0x3A000000
    hi_bits = np.float32(512.0).view(np.uint32)           # 0x44000000
    with ThreadPoolExecutor(ncores()) as ex:
        for first in range(0, 1 << 31, 1 << 28):
            n = 1 << 28
            pos = _encode(oracle_mod, first, n, ex)
            neg = _encode(oracle_mod, first | 0x80000000, n, ex)
            bits = np.arange(first, first + n, dtype=np.uint64).astype(np.uint32)
            nan = bits > 0x7F800000
            assert np.array_equal(neg[~nan], pos[~nan] | 0x80), hex(first)
            assert np.all(pos[nan] == 0x7F) and np.all((neg[nan] & 0x7F) == 0x7F), hex(first)
            small, big = bits < lo_bits, (bits >= hi_bits) & ~nan
            assert np.all(pos[small] == 0) and np.all(pos[big] == 0x7E), hex(first)
            mid = ~small & ~big & ~nan
            if mid.any():
                want = _nearest_codes(bits[mid])
                got = pos[mid]
                if not np.array_equal(got, want):
                    i = int(np.nonzero(got != want)[0][0])
                    raise AssertionError(f"0x{int(bits[mid][i]):08x}: oracle 0x{got[i]:02x}, "
                                         f"nearest 0x{want[i]:02x}")
