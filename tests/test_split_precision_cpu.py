"""The rounding identities the tensor-core kernels rely on, emulated on the CPU with the same
integer operations on fp32 bit patterns that the kernels use:

- round to nearest tf32 (10 explicit mantissa bits, ties away from zero): add half a tf32 ulp to
  the pattern and clear the 13 low bits; |error| <= 2^-11 |x|;
- the tensor core reads an fp32 operand as tf32 by dropping the 13 low mantissa bits, so
  x = hi + lo with hi = x truncated and lo = x - hi exact in fp32;
- bf16 hi + lo split by truncation (8 + 8 significant bits): |x - hi - lo| < 2^-15 |x|;
- three tf32 products hi*hi + hi*lo + lo*hi (each operand read truncated) reproduce an fp32
  dot product to about 2^-20 relative (the dropped lo*lo term and the truncation of lo).
"""
import numpy as np


def _bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def _f32(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


def tf32_round(x):
    return _f32((_bits(x) + np.uint32(0x1000)) & np.uint32(0xFFFFE000))


def tf32_trunc(x):
    return _f32(_bits(x) & np.uint32(0xFFFFE000))


def bf16_trunc(x):
    return _f32(_bits(x) & np.uint32(0xFFFF0000))


def _samples(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)


def test_round_to_nearest_tf32_is_within_half_an_ulp():
    x = _samples(200000, 1)
    r = tf32_round(x)
    err = np.abs(r.astype(np.float64) - x.astype(np.float64))
    assert np.all(err <= np.exp2(-11) * np.abs(x.astype(np.float64)))
    assert np.all((_bits(r) & np.uint32(0x1FFF)) == 0)  # exactly representable in tf32


def test_round_to_nearest_tf32_ties_away_from_zero():
    half_ulp = np.uint32(0x1000)
    base = _bits(np.float32(1.5)) & np.uint32(0xFFFFE000)
    x = _f32(np.array([base + half_ulp], dtype=np.uint32))  # exactly between two tf32 values
    assert tf32_round(x)[0] > x[0]
    assert tf32_round(-x)[0] < -x[0]


def test_truncation_split_is_exact():
    x = _samples(200000, 2)
    hi = tf32_trunc(x)
    lo = (x - hi).astype(np.float32)
    assert np.all(hi.astype(np.float64) + lo.astype(np.float64) == x.astype(np.float64))


def test_bf16_hi_lo_split_error():
    x = _samples(200000, 3)
    hi = bf16_trunc(x)
    lo = bf16_trunc((x - hi).astype(np.float32))
    err = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert np.all(err < np.exp2(-15) * np.abs(x.astype(np.float64)))


def test_three_tf32_products_reproduce_fp32_products():
    rng = np.random.Generator(np.random.PCG64(4))
    a = rng.standard_normal((64, 128)).astype(np.float32)
    b = rng.standard_normal((128, 32)).astype(np.float32)
    ah, bh = tf32_trunc(a), tf32_trunc(b)
    al, bl = tf32_trunc((a - ah).astype(np.float32)), tf32_trunc((b - bh).astype(np.float32))
    f = lambda u, w: u.astype(np.float64) @ w.astype(np.float64)  # noqa: E731
    split3 = f(ah, bh) + f(ah, bl) + f(al, bh)
    exact = f(a, b)
    scale = np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64)
    assert np.max(np.abs(split3 - exact) / scale) < np.exp2(-19)
    one = f(ah, bh)  # a single tf32 product is far less accurate
    assert np.max(np.abs(one - exact) / scale) > np.exp2(-14)
