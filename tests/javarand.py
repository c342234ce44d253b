"""java.util.Random, written from its published specification (the Java SE
API documentation of java.util.Random): a 48-bit linear congruential
generator with multiplier 0x5DEECE66D and addend 0xB; nextDouble joins 26 and
27 generated bits; nextGaussian is the polar method of Box, Muller and
Marsaglia, returning the two deviates of each accepted pair in turn;
nextInt(bound) rejects the biased tail.

Used only by the tests, to rebuild the seeded inputs of the Java examples in
"Building Q8_0 and Q4_0 Like ggml" (Examples 10-15), whose printed outputs pin
the oracle. It holds none of the quantization arithmetic.
"""
import math

import numpy as np

_MULT = 0x5DEECE66D
_ADD = 0xB
_MASK = (1 << 48) - 1


class JavaRandom:
    def __init__(self, seed: int):
        self.seed = (seed ^ _MULT) & _MASK
        self._next_gaussian = None

    def next_bits(self, bits: int) -> int:
        self.seed = (self.seed * _MULT + _ADD) & _MASK
        r = self.seed >> (48 - bits)
        # Java returns the low 32 bits as a signed int
        r &= 0xFFFFFFFF
        return r - (1 << 32) if r >= (1 << 31) else r

    def next_int(self, bound: int) -> int:
        if bound <= 0:
            raise ValueError("bound must be positive")
        if bound & (bound - 1) == 0:
            return (bound * self.next_bits(31)) >> 31
        while True:
            bits = self.next_bits(31)
            val = bits % bound
            # Java's overflow test: bits - val + (bound - 1) < 0 as int32
            t = bits - val + (bound - 1)
            if t < (1 << 31):
                return val

    def next_double(self) -> float:
        return ((self.next_bits(26) << 27) + self.next_bits(27)) * (1.0 / (1 << 53))

    def next_gaussian(self) -> float:
        if self._next_gaussian is not None:
            g, self._next_gaussian = self._next_gaussian, None
            return g
        while True:
            v1 = 2 * self.next_double() - 1
            v2 = 2 * self.next_double() - 1
            s = v1 * v1 + v2 * v2
            if 0 < s < 1:
                break
        multiplier = math.sqrt(-2 * math.log(s) / s)
        self._next_gaussian = v2 * multiplier
        return v1 * multiplier


def f32(v) -> np.float32:
    """Java's (float) cast of a double: round to nearest f32."""
    return np.float32(v)
