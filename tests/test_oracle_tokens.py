"""Pins of the oracle's 1 x 128 activation codec (MoE dispatch) against
exact-rational brute force, the dequantisation error bound, and the
invariance of codes under power-of-two scaling of a group."""
from fractions import Fraction

import numpy as np
import pytest

import bruteforce as bf


def _bits(rng, shape, sigma=0.02, zero_rows=(), outliers=0):
    x = rng.standard_t(3, size=shape).astype(np.float32) * np.float32(sigma)
    b = (x.view(np.uint32) >> 16).astype(np.uint16)          # truncation is fine: any BF16 will do
    for r in zero_rows:
        b[r] = 0
    for _ in range(outliers):
        r, c = rng.integers(0, shape[0]), rng.integers(0, shape[1])
        b[r, c] = 0x46EA if rng.integers(0, 2) else 0xC6EA     # +-29952
    return b


@pytest.mark.parametrize("shape", [(1, 1), (3, 130), (2, 128), (4, 300), (1, 7)])
def test_tokens_match_exact_rational_brute_force(oracle_mod, shape):
    rng = np.random.default_rng(sum(shape))
    b = _bits(rng, shape, zero_rows=(0,) if shape[0] > 2 else (), outliers=2)
    if shape[1] > 2:
        b[-1, 0] = 0x8000                                   # -0.0
        b[-1, 1] = 0x0001                                   # a BF16 subnormal
    codes, scales = oracle_mod.quantize_tokens(b)
    want_c, want_s = bf.quantize_rows(b.ravel().tolist(), *shape)
    assert codes.ravel().tolist() == want_c
    assert [Fraction(float(v)) for v in scales.ravel()] == want_s


def test_tokens_subnormal_scale_group(oracle_mod):
    b = np.zeros((1, 128), np.uint16)
    b[0, :5] = [0x0001, 0x8002, 0x0003, 0x0000, 0x8000]     # amax = 3 * 2^-133
    codes, scales = oracle_mod.quantize_tokens(b)
    want_c, want_s = bf.quantize_rows(b.ravel().tolist(), 1, 128)
    assert codes.ravel().tolist() == want_c and Fraction(float(scales[0, 0])) == want_s[0]


def test_tokens_dequantisation_error_bound(oracle_mod):
    rng = np.random.default_rng(7)
    b = _bits(rng, (64, 7168), outliers=20)
    codes, scales = oracle_mod.quantize_tokens(b)
    x = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dec = np.array([oracle_mod.e4m3_decode(c) for c in range(256)])
    s = np.repeat(scales.astype(np.float64), 128, axis=1)[:, :7168]
    q = dec[codes]
    y = np.abs(x / s)
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    ulp = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    assert np.all(np.abs(x - q * s) <= (ulp / 2 + y * 2.0 ** -24) * s + 1e-300)


def test_tokens_strided_rows_equal_contiguous(oracle_mod):
    rng = np.random.default_rng(11)
    wide = _bits(rng, (5, 400))
    codes_s, scales_s = oracle_mod.quantize_tokens(wide[:, :260])       # ld 400, hidden 260
    codes_c, scales_c = oracle_mod.quantize_tokens(np.ascontiguousarray(wide[:, :260]))
    assert np.array_equal(codes_s, codes_c) and np.array_equal(scales_s, scales_c)


def test_tokens_power_of_two_scaling_invariance(oracle_mod):
    """Scaling a group by 2^k scales its scale by exactly 2^k and leaves every
    code unchanged (no overflow, no subnormal scale)."""
    rng = np.random.default_rng(13)
    b = _bits(rng, (8, 512), outliers=3)
    codes, scales = oracle_mod.quantize_tokens(b)
    for k in (-20, -3, 1, 17):
        exp = ((b >> 7) & 0xFF).astype(np.int32)
        nz = exp > 0
        assert np.all(exp[nz] + k > 0) and np.all(exp[nz] + k < 255)
        b2 = b.copy()
        b2[nz] = ((b[nz] & 0x807F) | (((exp[nz] + k) & 0xFF) << 7)).astype(np.uint16)
        codes2, scales2 = oracle_mod.quantize_tokens(b2)
        assert np.array_equal(codes2, codes)
        assert np.array_equal(scales2, np.ldexp(scales, k).astype(np.float32))
