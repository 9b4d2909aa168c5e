"""bf16 helpers of the oracle (test infrastructure only).

bf16 is the top 16 bits of an IEEE binary32.  ``decode`` widens bit patterns to fp64
exactly; ``round_rne`` rounds fp64 values to the nearest bf16 value (ties to even), going
through binary32 first only when that cannot double-round: it rounds fp64 straight to an
8-bit significand with ``np.frexp`` / ``np.ldexp``.
"""
from __future__ import annotations

import numpy as np


def decode(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_rne(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16-representable value (ties to even), as fp64.

    Written from the definition: a bf16 normal number has an 8-bit significand, so
    v = m * 2^e with 0.5 <= |m| < 1 rounds to rint(m * 2^8) * 2^(e-8); ``np.rint`` rounds
    half to even.  Values below the smallest normal bf16 (2^-126) round on the subnormal
    grid of spacing 2^-133.  Overflow past the largest finite bf16 gives +-inf.
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    e = np.maximum(e, -125)           # subnormal grid: spacing 2^(-125-8) = 2^-133
    r = np.ldexp(np.rint(np.ldexp(v, 8 - e)), e - 8)
    big = np.abs(r) > 3.3895313892515355e38
    if np.any(big):
        r = np.where(big, np.sign(r) * np.inf, r)
    return r


def to_bits(v: np.ndarray) -> np.ndarray:
    """fp64 values that are exactly bf16-representable -> uint16 bit patterns."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
