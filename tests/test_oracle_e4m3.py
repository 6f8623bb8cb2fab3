"""Pins of the oracle's e4m3 encoder/decoder against things other than
itself: torch's float8_e4m3fn (a library routine), an exact-rational
nearest-code search, and values fixed by the format definition."""
import numpy as np
import pytest
import torch

import bruteforce as bf


def test_decode_matches_torch_for_all_256_codes(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for c in range(256):
        got = oracle_mod.e4m3_decode(c)
        want = float(ref[c])
        if np.isnan(want):
            assert np.isnan(got) and (c & 0x7F) == 0x7F
        else:
            assert got == want and np.signbit(got) == np.signbit(want), hex(c)


def test_format_landmarks(oracle_mod):
    # largest finite, smallest normal, smallest subnormal, one, signed zero
    enc = oracle_mod.e4m3_encode
    assert enc([448.0])[0] == 0x7E and enc([-448.0])[0] == 0xFE
    assert enc([2.0 ** -6])[0] == 0x08
    assert enc([2.0 ** -9])[0] == 0x01
    assert enc([1.0])[0] == 0x38
    assert enc([0.0])[0] == 0x00 and enc([-0.0])[0] == 0x80
    assert enc([np.nan])[0] == 0x7F
    assert enc([np.float32(-np.nan)])[0] == 0xFF
    # saturation instead of NaN above the largest finite value
    for v in (448.5, 463.9, 464.0, 470.0, 480.0, 1e30, np.inf):
        assert enc([v])[0] == 0x7E and enc([-v])[0] == 0xFE


def test_encode_decode_identity_on_all_finite_codes(oracle_mod):
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        v = oracle_mod.e4m3_decode(c)
        assert oracle_mod.e4m3_encode([v])[0] == c, hex(c)


def _stratified_values():
    """Every binade from 2^-14 to 2^9, each e4m3 rounding boundary of every
    binade +-3 fp32 ulps, plus random mantissas, both signs."""
    rng = np.random.default_rng(7)
    out = []
    for e in range(-14, 10):
        base = np.float32(2.0 ** e)
        bits = int(np.float32(base).view(np.uint32))
        mants = list(rng.integers(0, 1 << 23, 64))
        for k in range(0, 1 << 23, 1 << 19):          # every multiple of the 4th-bit step
            for d in (-3, -2, -1, 0, 1, 2, 3):
                mants.append((k + d) % (1 << 23))
        for m in mants:
            out.append(bits + int(m))
    arr = np.array(sorted(set(out)), dtype=np.uint32)
    return np.concatenate([arr, arr | np.uint32(0x80000000)]).view(np.float32)


def test_encode_matches_exact_nearest_search(oracle_mod):
    ys = _stratified_values()
    got = oracle_mod.e4m3_encode(ys)
    for y, g in zip(ys.tolist(), got.tolist()):
        want = bf.nearest_code(bf.Fraction(y), negative_zero=np.signbit(y))
        assert g == want, (y, hex(g), hex(want))


def test_encode_matches_torch_over_every_nonsaturating_fp32(oracle_mod):
    """Exhaustive over all fp32 bit patterns with magnitude in [2^-11, 464]
    (below 2^-11 every value encodes to a signed zero, checked next)."""
    lo = int(np.float32(2.0 ** -11).view(np.uint32))
    hi = int(np.float32(464.0).view(np.uint32)) + 1
    step = 1 << 23
    for sign in (0, 0x80000000):
        for first in range(lo, hi, step):
            n = min(step, hi - first)
            got = oracle_mod.e4m3_encode_bits_range(first | sign, n)
            bits = np.arange(first, first + n, dtype=np.uint32) | np.uint32(sign)
            want = torch.from_numpy(bits.view(np.float32)).to(torch.float8_e4m3fn)
            want = want.view(torch.uint8).numpy()
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, (hex(int(bits[bad[0]])), got[bad[0]], want[bad[0]])


def test_encode_tiny_and_huge_ranges(oracle_mod):
    rng = np.random.default_rng(11)
    # |y| < 2^-11: always signed zero
    top = int(np.float32(2.0 ** -11).view(np.uint32))
    b = np.concatenate([rng.integers(0, top, 2_000_000, dtype=np.uint32),
                        np.arange(0, 4096, dtype=np.uint32),
                        np.arange(top - 4096, top, dtype=np.uint32)])
    for sign in (0, 0x80000000):
        got = oracle_mod.e4m3_encode((b | np.uint32(sign)).view(np.float32))
        assert np.all(got == (0x80 if sign else 0))
    # |y| > 464 including inf: saturates
    lo = int(np.float32(464.0).view(np.uint32)) + 1
    inf = 0x7F800000
    b = np.concatenate([rng.integers(lo, inf, 2_000_000, dtype=np.uint32),
                        np.array([lo, inf], dtype=np.uint32)])
    for sign in (0, 0x80000000):
        got = oracle_mod.e4m3_encode((b | np.uint32(sign)).view(np.float32))
        assert np.all(got == (0xFE if sign else 0x7E))
    # NaNs keep their sign
    nans = rng.integers(inf + 1, 0x80000000, 100_000, dtype=np.uint32)
    assert np.all(oracle_mod.e4m3_encode(nans.view(np.float32)) == 0x7F)
    assert np.all(oracle_mod.e4m3_encode((nans | np.uint32(0x80000000)).view(np.float32)) == 0xFF)


def test_ties_go_to_even_at_every_midpoint(oracle_mod):
    vals = [bf.E4M3_VALUES[i] for i in range(len(bf.E4M3_VALUES))]
    for i in range(len(vals) - 1):
        mid = (vals[i] + vals[i + 1]) / 2
        if float(mid) != mid:
            continue          # midpoint not representable in fp32 (never here)
        got = oracle_mod.e4m3_encode([float(mid)])[0]
        assert got == (i if i % 2 == 0 else i + 1), (float(mid), got)
