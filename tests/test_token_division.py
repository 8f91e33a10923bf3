"""The prologue kernel finds a row's token as t = (r * magic) >> shift instead of r / H.

The host picks shift = 31 + ceil(log2 H) and magic = ceil(2^shift / H); the kernel multiplies a 32-bit
row index (r < 2^31) by a 32-bit magic. This checks the rule itself: magic fits 32 bits for every
head count, and the quotient is exact over the whole row range (both ends, every multiple of H
and its neighbours near the top, and random rows).
"""
import numpy as np
import pytest


def magic_for(h: int):
    lg = 0
    while (1 << lg) < h:
        lg += 1
    shift = 31 + lg
    return ((1 << shift) + h - 1) // h, shift


HEADS = list(range(1, 257)) + [320, 384, 511, 512, 513, 1000, 1024, 4095, 4096, 4097, 65535, 65536]


@pytest.mark.parametrize("h", HEADS)
def test_magic_fits_32_bits_and_divides_exactly(h):
    magic, shift = magic_for(h)
    assert magic < 2**32
    rng = np.random.default_rng(h)
    top = 2**31 - 1
    r = np.concatenate([
        np.arange(0, min(4 * h + 8, top), dtype=np.uint64),
        np.arange(top - 4 * h - 8, top + 1, dtype=np.uint64),
        (np.arange(1, 2000, dtype=np.uint64) * np.uint64(top // 2000 // h * h)),
        rng.integers(0, top + 1, size=20000, dtype=np.uint64),
    ])
    r = r[r <= top]
    got = (r * np.uint64(magic)) >> np.uint64(shift)  # r < 2^31, magic < 2^32: no uint64 overflow
    assert np.array_equal(got, r // np.uint64(h))
    # multiples of h and the row just before each, near the top of the range
    m = (np.uint64(top) // np.uint64(h) - np.arange(0, 64, dtype=np.uint64)) * np.uint64(h)
    for rr in (m, m - np.uint64(1)):
        rr = rr[rr <= top]
        assert np.array_equal((rr * np.uint64(magic)) >> np.uint64(shift), rr // np.uint64(h))
