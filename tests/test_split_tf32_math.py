"""The arithmetic behind the split-tf32 products of the RWKV-8 kernels
(csrc/rwkv8_split.cuh), emulated bit for bit in numpy on the host.

tf32 keeps 10 explicit mantissa bits of an fp32 pattern. The kernels round x
to tf32 by adding half a tf32 unit (bit 12) to the pattern and clearing the 13
low bits, take lo = x - hi in fp32 and round lo the same way, and form a b as
a_hi b_hi + a_hi b_lo + a_lo b_hi. Checked here: hi is a tf32 value and the
nearest one (|x - hi| <= 2^-11 |x|, ties away from zero); x - hi is exact in
fp32; and the three products miss a b by at most 2^-20 |a b|, far inside the
fp32 parity bar of 1e-4 (1 + |ref|) that the GPU tests hold the kernels to.
"""
import numpy as np


def tf32_round(x32):
    bits = x32.view(np.uint32)
    return ((bits + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def split(x32):
    hi = tf32_round(x32)
    lo = tf32_round((x32 - hi).astype(np.float32))
    return hi, lo


def _samples(n, seed):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(-1.0, 1.0, n)
    expo = rng.integers(-60, 60, n)
    return (mant * np.exp2(expo)).astype(np.float32)


def test_hi_is_the_nearest_tf32_value():
    x = _samples(200_000, 1)
    hi = tf32_round(x)
    assert np.all(hi.view(np.uint32) & np.uint32(0x1FFF) == 0)
    rel = np.abs(x.astype(np.float64) - hi.astype(np.float64)) / np.abs(x.astype(np.float64))
    assert rel.max() <= 2.0 ** -11
    # nearest: the tf32 neighbour on the other side is never closer
    step = np.exp2(np.floor(np.log2(np.abs(hi.astype(np.float64)))) - 10)
    other = hi.astype(np.float64) - np.sign(x.astype(np.float64) - hi.astype(np.float64)) * step
    assert np.all(np.abs(x - hi.astype(np.float64)) <= np.abs(x - other) + 1e-300)


def test_remainder_is_exact_in_fp32():
    x = _samples(200_000, 2)
    hi = tf32_round(x)
    lo32 = (x - hi).astype(np.float32)
    assert np.array_equal(lo32.astype(np.float64), x.astype(np.float64) - hi.astype(np.float64))


def test_three_products_reach_fp32_accuracy():
    a, b = _samples(200_000, 3), _samples(200_000, 4)
    ah, al = split(a)
    bh, bl = split(b)
    f = lambda u: u.astype(np.float64)  # noqa: E731  (tf32 products are exact in fp64)
    approx = f(ah) * f(bh) + f(ah) * f(bl) + f(al) * f(bh)
    exact = f(a) * f(b)
    rel = np.abs(approx - exact) / np.abs(exact)
    assert rel.max() <= 2.0 ** -20
    one = f(ah) * f(bh)  # a single tf32 product, for contrast
    assert (np.abs(one - exact) / np.abs(exact)).max() > 2.0 ** -13
