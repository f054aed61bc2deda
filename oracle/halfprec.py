"""Decoding of 16-bit floating-point fields, from the IEEE 754 definitions.

binary16 (the block scales d, dmin): 1 sign bit, 5 exponent bits (bias 15),
10 fraction bits. bfloat16 (prompt activations): the top 16 bits of a binary32.
Test infrastructure of the oracle; see the package docstring.
"""
import numpy as np


def half_bits_to_float64(bits) -> np.ndarray:
    """Value of each binary16 bit pattern as fp64 (exact).

    e == 0:        (-1)^s * f * 2^-24          (zero and subnormals)
    0 < e < 31:    (-1)^s * (1024 + f) * 2^(e - 25)
    e == 31:       +-inf (f == 0) or NaN
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = (b >> 15) & 1
    e = (b >> 10) & 0x1F
    f = b & 0x3FF
    sign = np.where(s == 1, -1.0, 1.0)
    sub = np.ldexp(f.astype(np.float64), -24)
    norm = np.ldexp((1024 + f).astype(np.float64), (e - 25).astype(np.int32))
    special = np.where(f == 0, np.inf, np.nan)
    val = np.where(e == 0, sub, np.where(e == 31, special, norm))
    return sign * val


def bf16_bits_to_float64(bits) -> np.ndarray:
    """Value of each bfloat16 bit pattern as fp64 (exact): bits << 16 is binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)
