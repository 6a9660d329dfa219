"""The multiply-shift division the kernels use for every fixed divisor
(tile decode, pixel -> (image, row, column), the gather loader's runs):
q = (umulhi(x, mul) + x) >> shift with shift = ceil(log2 d) and
mul = floor(2^32 * (2^shift - d) / d) + 1 (mod 2^32), exact for 0 <= x < 2^31.

This checks the arithmetic itself (written out here from that definition)
against Python's integer division; the GPU parity tests exercise the kernels
that use it.
"""
import random

import pytest


def _params(d):
    shift = (d - 1).bit_length()            # ceil(log2 d); 0 for d = 1
    mul = ((1 << 32) * ((1 << shift) - d) // d + 1) & 0xFFFFFFFF
    return mul, shift


def _div(x, mul, shift):
    hi = (x * mul) >> 32                     # umulhi of two 32-bit values
    return (hi + x) >> shift                 # the sum fits in 33 bits: no wrap


def _edge_values(d):
    top = (1 << 31) - 1
    vals = {0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, top, top - 1, top - d}
    k = top // d
    vals |= {k * d - 1, k * d, min(top, k * d + d - 1)}
    return [v for v in vals if 0 <= v <= top]


@pytest.mark.parametrize("d", list(range(1, 600)) + [
    1000, 1023, 1024, 1025, 3136, 12544, 25088, 100352, 401408, 65535, 65536, 65537,
    (1 << 20) - 1, 1 << 20, (1 << 20) + 1, 999983, (1 << 30) - 1, 1 << 30, (1 << 31) - 1])
def test_multiply_shift_division_is_exact(d):
    mul, shift = _params(d)
    rng = random.Random(d)
    xs = _edge_values(d) + [rng.randrange(0, 1 << 31) for _ in range(200)]
    for x in xs:
        assert _div(x, mul, shift) == x // d, (d, x)
