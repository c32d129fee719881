"""bfloat16 codec for the oracle, written from the IEEE 754 definition.

bfloat16 keeps float32's 8-bit exponent and 8 significant bits (7 stored).
``round_bf16`` rounds a float64 value *directly* to the nearest bfloat16 with
ties to even; it never passes through float32, because float64 -> float32 ->
bfloat16 can round twice and land on the wrong neighbour.

Rounding points are where the pages put them: the Gaudi cookbook port of
Beam-1.0 ("What was built -> Model code") says the reference rounds to bf16
after the sandwich norms and the depth-scaled residuals, and the vLLM Beam
summary (kernel change 1) keeps "FP32 math and the reference's BF16 rounding
points".
"""
from __future__ import annotations

import numpy as np

# largest finite bfloat16: (2 - 2**-7) * 2**127
BF16_MAX = float.fromhex("0x1.fep127")
# exponent of the smallest normal bfloat16 (same as float32)
_EMIN = -126
_PREC = 8  # significant bits


def decode(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def round_bf16(v) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    For a finite v with frexp exponent ex (v = m * 2**ex, 0.5 <= |m| < 1) the
    spacing of bfloat16 values around v is 2**(ex - 8) in the normal range and
    the fixed 2**(-133) below 2**-126. Dividing by that spacing is exact (a
    power of two), ``np.rint`` rounds half to even, and multiplying back is
    exact. Results above the largest finite value become +-inf; NaN stays NaN.
    """
    v = np.asarray(v, dtype=np.float64)
    _, ex = np.frexp(v)
    eq = np.maximum(ex, _EMIN + 1) - _PREC
    r = np.ldexp(np.rint(np.ldexp(v, -eq)), eq)
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, v), r)
    return np.where(np.isfinite(v), r, v)


def encode(v) -> np.ndarray:
    """float64 values -> bf16 bit patterns after rounding with ``round_bf16``."""
    r = round_bf16(v).astype(np.float32)  # exact: every bfloat16 is a float32
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def ulp_distance(a_bits, b_bits) -> np.ndarray:
    """Number of representable bfloat16 steps between two bit patterns.

    Bit patterns are mapped to a monotone integer line (sign-magnitude to
    two's complement); +0 and -0 both map to 0."""
    def ordered(bits):
        b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordered(a_bits) - ordered(b_bits))
