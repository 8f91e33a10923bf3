"""Row-length divisions on the device: x / n for a power-of-two n is taken as x * (1/n).

The kernels recognise a power of two from the float's bit pattern (zero mantissa field), form 1/n
as the bit pattern 0x7f000000 - bits(n), and multiply. This checks that rule in IEEE fp32 on the
host: the reciprocal is exact, and the rounded product equals the rounded quotient for every
power-of-two row length the kernels meet, over normal, subnormal, zero and signed inputs.
"""
import numpy as np
import pytest


def recip_bits(n: np.float32) -> np.float32:
    b = np.array([n], dtype=np.float32).view(np.uint32)[0]
    return np.array([np.uint32(0x7F000000) - b], dtype=np.uint32).view(np.float32)[0]


def is_pow2_bits(n: np.float32) -> bool:
    return (int(np.array([n], dtype=np.float32).view(np.uint32)[0]) & 0x7FFFFF) == 0


@pytest.mark.parametrize("k", range(0, 25))
def test_power_of_two_reciprocal_and_quotient(k):
    n = np.float32(2.0 ** k)
    assert is_pow2_bits(n)
    r = recip_bits(n)
    assert r == np.float32(1.0) / n and float(r) == 2.0 ** -k  # exact reciprocal
    rng = np.random.default_rng(k)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(1e3),
        rng.random(1000).astype(np.float32) * np.float32(1e-36),  # results reach the subnormal range
        np.array([0.0, -0.0, 1.0, -1.0, np.finfo(np.float32).max, np.finfo(np.float32).tiny,
                  np.float32(1.4e-45)], dtype=np.float32),
    ])
    with np.errstate(under="ignore"):
        prod = x * r
        quot = x / n
    assert np.array_equal(prod.view(np.uint32), quot.view(np.uint32))  # bit for bit, signed zeros too


@pytest.mark.parametrize("n", [3.0, 96.0, 192.0, 1000.0, 1536.0, 3072.0, 4095.0])
def test_other_lengths_take_the_division(n):
    assert not is_pow2_bits(np.float32(n))
