"""The two facts of fp16 arithmetic that the fp16 combine kernels rest on,
checked on the CPU with numpy's IEEE fp16 / fp32 / fp64.

1. Widening by x + (-0): every finite fp16 number x is an fp32 number, and
   x + (-0) = x bit for bit, -0 and subnormals included.
2. A product of two fp16 numbers is exact in fp32 (11 + 11 significant bits
   fit in fp32's 24, and the product's exponent range, from 2^-48 up to
   65504^2 < 2^32, lies inside fp32's normal range), so fma(a, b, c) in fp32
   rounds once whether a and b are fp16 or their fp32 widenings: the kernel
   that multiplies fp16 rows by fp16 weights without widening them gives the
   widening kernel's bits."""
import numpy as np


def _finite_f16():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = codes.view(np.float16)
    return codes[np.isfinite(x)], x[np.isfinite(x)]


def test_adding_negative_zero_widens_every_fp16_exactly():
    codes, x = _finite_f16()
    assert codes.size == 63488
    wide = x.astype(np.float32)
    assert np.array_equal(wide.astype(np.float16).view(np.uint16), codes)  # fp16 -> fp32 is exact
    summed = wide + np.float32(-0.0)
    assert np.array_equal(summed.view(np.uint32), wide.view(np.uint32))    # x + (-0) = x, -0 kept


def test_fp16_products_are_exact_in_fp32():
    _, x = _finite_f16()
    rng = np.random.Generator(np.random.PCG64(1616))
    a = rng.choice(x, 2_000_000)
    b = rng.choice(x, 2_000_000)
    # the subnormals and the largest binade (every fourth code, plus the
    # endpoints 2^-24, the largest subnormal, 2^-14 and 65504), all against all
    sub = x[np.abs(x.astype(np.float64)) < 2.0 ** -14]
    top = x[np.abs(x) >= 32768]
    edge = np.array([2.0 ** -24, 1023 * 2.0 ** -24, 2.0 ** -14, 65504.0], np.float16)
    ends = np.concatenate([sub[::4], top[::4], edge, -edge])
    a = np.concatenate([a, np.repeat(ends, ends.size)])
    b = np.concatenate([b, np.tile(ends, ends.size)])
    p32 = a.astype(np.float32) * b.astype(np.float32)
    p64 = a.astype(np.float64) * b.astype(np.float64)
    assert np.array_equal(p32.astype(np.float64), p64)
    assert np.all(np.abs(p64[p64 != 0]) >= 2.0 ** -48) and np.all(np.abs(p64) < 2.0 ** 32)
