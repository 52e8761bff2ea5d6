"""TF32 rounding on the host, for tests of the prefill's operand rounding.

TF32 keeps float32's sign and 8-bit exponent and 10 of its 23 fraction bits.
`rna_exact` rounds to that grid from the definition (exact rational arithmetic,
round to nearest, ties away from zero, overflow to infinity); `add_half_bits`
is the bit-level method the prefill uses (add half a TF32 unit in the last place
to the bit pattern and let the low 13 bits be dropped).
"""
from fractions import Fraction
import math

import numpy as np

LOW = np.uint32(0x1FFF)


def rna_exact(bits: int) -> int:
    """Round the float32 with these bits to TF32 (ties away), by definition; returns f32 bits."""
    bits = int(bits) & 0xFFFFFFFF
    sign = bits & 0x80000000
    x = float(np.uint32(bits).view(np.float32))
    if math.isnan(x):
        return 0x7FFFFFFF
    a = abs(x)
    if math.isinf(a) or a == 0.0:
        return bits
    _, e2 = math.frexp(a)                 # a = m * 2^e2, m in [0.5, 1)
    e = max(e2 - 1, -126)                 # binade of a (subnormals share the smallest one)
    u = Fraction(2) ** (e - 10)           # TF32 unit in the last place
    q = math.floor(Fraction(a) / u + Fraction(1, 2)) * u
    if q >= Fraction(2) ** 128:
        return sign | 0x7F800000
    return sign | int(np.float32(float(q)).view(np.uint32))


def add_half_bits(b: np.ndarray) -> np.ndarray:
    """The bit pattern read as a signed 32-bit integer, plus 2^12 with wrap-around, then the
    signed maximum of that and the input (a positive NaN that would carry into the sign bit
    is kept as it is); uint32 array in and out."""
    s = np.asarray(b, np.uint32).view(np.int32).astype(np.int64)
    t = (s + 0x1000 + 2 ** 31) % 2 ** 32 - 2 ** 31
    return (np.maximum(t, s) % 2 ** 32).astype(np.uint32)


def rna_array(x: np.ndarray) -> np.ndarray:
    """float32 array rounded to TF32 (ties away) by the bit method, low bits cleared."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    return (add_half_bits(b) & ~LOW).view(np.float32)


def sweep_bits(n_random: int = 20000, seed: int = 7) -> np.ndarray:
    """Every exponent with mantissas at and around the rounding boundary, both signs, the
    special values, and random patterns (uint32)."""
    lows = [0x0, 0x1, 0xFFF, 0x1000, 0x1001, 0x1FFF]
    highs = [0x0, 0x1, 0x155, 0x2AA, 0x3FE, 0x3FF]
    out = [(s << 31) | (e << 23) | (h << 13) | lo
           for s in (0, 1) for e in range(255) for h in highs for lo in lows]
    out += [0x7F800000, 0xFF800000, 0x7FC00000, 0x7FFFFFFF, 0xFFFFFFFF, 0x7F800001, 0x7FFFF000,
            0xFFFFF000, 0x00000000, 0x80000000, 0x7F7FFFFF, 0x7F7FF000, 0x7F7FEFFF]
    rnd = np.random.default_rng(seed).integers(0, 2 ** 32, size=n_random, dtype=np.uint64)
    return np.concatenate([np.array(out, np.uint64), rnd]).astype(np.uint32)
