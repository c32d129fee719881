"""NVFP4 experts: 4-bit E2M1 values with an E4M3 scale per 16 values and an
FP32 scale on top, for the expert weights and (at runtime) the expert inputs.

This module is test infrastructure: only the tests, the smoke check and the
benchmark's CPU legs use it. It shares no code with the CUDA path.

Sources:
* TokenSpeed blog, "Model architecture and precision -> NVFP4 and FP8
  checkpoints": the NVFP4 checkpoint quantizes only the expert weights; each
  weight is a 4-bit float (E2M1), every 16 weights share an FP8 (E4M3) scale,
  and each expert has an additional FP32 scale. Expert inputs are quantized
  in the same format at runtime, so the expert GEMMs run as FP4 x FP4.
* Same page, "TensorRT-LLM NVFP4 MoE": input quantization does not depend on
  routing; the kernel takes NVFP4 inputs and reads about a quarter of the
  weight bytes of BF16.

The two element formats, written out from their definitions:
* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
  0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6; no infinity or NaN. Code bit 3 is
  the sign.
* E4M3 ("fn" variant): sign, 4 exponent bits (bias 7), 3 mantissa bits;
  subnormals in steps of 2**-9; largest finite 448; codes 0x7F and 0xFF are
  NaN; no infinity.

Readings taken where the pages give the format but not the recipe:
* a block is 16 consecutive values along the reduction (K) dimension of one
  row (a weight row, or one token's activation row);
* with the FP32 scale g, a block's scale is s = E4M3(amax / (6 g)) and each
  value's code is q = E2M1(x / (s g)); both roundings are to nearest with ties
  to the even code and saturate at the largest finite value (6 and 448); a
  block with s = 0 has all codes 0. The value represented is q * s * g;
* these decisions are taken in FP32 arithmetic (6 g, amax / (6 g), s g and
  x / (s g) each rounded to FP32), the precision of the GPU path;
* the FP32 scale of an expert is one number for all three of its matrices:
  the largest |w| over its gate, up and down weights divided by 6 * 448, so
  the block holding that weight gets the largest E4M3 scale;
* the FP32 scales of the two activations (the expert input z and the SwiGLU
  output that feeds the down GEMM) are constants the caller passes (the role
  of a checkpoint's calibrated input scales);
* the products are accumulated without rounding here (float64); SiLU and the
  gate/up product are evaluated in float64 and rounded to FP32 before the
  SwiGLU output is quantized.
"""
from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


# ---------------------------------------------------------------- element formats
def e2m1_decode(codes) -> np.ndarray:
    """E2M1 codes (0..15) -> float64 values."""
    c = np.asarray(codes).astype(np.int64)
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.ldexp(1.0, (e - 1).astype(np.int64)))
    return np.where(c & 8, -mag, mag)


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 ("fn") codes (0..255) -> float64 values (NaN for 0x7F and 0xFF)."""
    c = np.asarray(codes).astype(np.int64)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64)))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


_E2M1_MAGS = e2m1_decode(np.arange(8))          # codes 0..7
_E4M3_MAGS = e4m3_decode(np.arange(0x7F))       # finite non-negative codes 0..126


def _nearest_even(a: np.ndarray, mags: np.ndarray) -> np.ndarray:
    """Index of the value in ``mags`` (ascending) nearest to each a >= 0,
    ties to the even index (the code whose last mantissa bit is 0); values
    above the largest saturate to it."""
    a = np.minimum(np.asarray(a, dtype=np.float64), mags[-1])
    hi = np.searchsorted(mags, a, side="left")          # first value >= a
    np.minimum(hi, mags.size - 1, out=hi)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - mags[lo], mags[hi] - a
    # the nearer neighbour; at equal distance the one with the even index
    # (of two neighbours exactly one is even: the upper one when lo is odd)
    take_hi = (dhi < dlo) | ((dhi == dlo) & (lo % 2 == 1))
    return np.where(take_hi, hi, lo)


def e2m1_round(v) -> np.ndarray:
    """Nearest E2M1 code of each value (ties to even, saturating at +-6). The
    sign bit is the value's, as in IEEE rounding: a negative value that
    rounds to zero gives -0 (code 8)."""
    v = np.asarray(v, dtype=np.float64)
    code = _nearest_even(np.abs(v), _E2M1_MAGS).astype(np.uint8)
    code |= np.signbit(v).astype(np.uint8) << 3
    return code


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 code of each non-negative value (ties to even, saturating at 448)."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(v < 0) or np.any(np.isnan(v)):
        raise ValueError("block scales are non-negative")
    return _nearest_even(v, _E4M3_MAGS).astype(np.uint8)


# ---------------------------------------------------------------- blocks of 16
BLOCK = 16


def quantize(x, g: float):
    """Quantize rows x [rows][K] (values exact in FP32) with FP32 scale g.

    Returns (codes uint8 [rows][K] in 0..15, scales uint8 [rows][K/16] E4M3
    codes). Every step is an FP32 operation, in the order of the reading in
    the module docstring."""
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % BLOCK:
        raise ValueError("rows of a multiple of 16 values expected")
    g = np.float32(g)
    rows, K = x.shape
    xb = x.reshape(rows, K // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=-1)                                   # exact
    s_code = e4m3_round(amax / (np.float32(6.0) * g))                # fp32 product, fp32 quotient
    s = e4m3_decode(s_code).astype(np.float32)
    d = (s * g)[..., None]                                           # fp32 product
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(d > 0, xb / np.where(d > 0, d, np.float32(1)), np.float32(0))  # fp32 quotient
    codes = e2m1_round(ratio.astype(np.float32))
    return codes.reshape(rows, K), s_code


def dequantize(codes, scales, g: float) -> np.ndarray:
    """Values q * s * g in float64 (exact: every factor is an FP32 value)."""
    codes = np.asarray(codes)
    rows, K = codes.shape
    s = e4m3_decode(scales).reshape(rows, K // BLOCK, 1)
    q = e2m1_decode(codes).reshape(rows, K // BLOCK, BLOCK)
    return (q * s * float(np.float32(g))).reshape(rows, K)


def pack_codes(codes) -> np.ndarray:
    """[rows][K] codes -> [rows][K/2] bytes, element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    """Inverse of pack_codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], 2 * p.shape[1]), dtype=np.uint8)
    out[:, 0::2] = p & 15
    out[:, 1::2] = p >> 4
    return out


# ---------------------------------------------------------------- experts
def expert_scale(Wg, Wu, Wd) -> np.float32:
    """An expert's FP32 scale: its largest |weight| over gate, up and down,
    divided by 6 * 448 (FP32 division)."""
    amax = max(float(np.abs(np.asarray(m, dtype=np.float32)).max()) for m in (Wg, Wu, Wd))
    return np.float32(amax) / np.float32(E2M1_MAX * E4M3_MAX)


class Nvfp4Expert:
    """One expert's NVFP4 weights: codes and block scales of gate [F][H],
    up [F][H] and down [H][F], and the expert's FP32 scale g."""

    def __init__(self, Wg, Wu, Wd, g=None):
        self.g = expert_scale(Wg, Wu, Wd) if g is None else np.float32(g)
        self.gate = quantize(Wg, self.g)
        self.up = quantize(Wu, self.g)
        self.down = quantize(Wd, self.g)

    def values(self):
        """(gate, up, down) as float64 values."""
        return tuple(dequantize(c, s, self.g) for c, s in (self.gate, self.up, self.down))


def silu(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def ffn(X, expert: Nvfp4Expert, g_in: float, g_act: float, return_act: bool = False):
    """One expert's NVFP4 SwiGLU FFN on rows X [n][H] (bf16 values).

    X is quantized with scale g_in; gate and up use the dequantized weights;
    a = silu(gate) * up is rounded to FP32 and quantized with scale g_act;
    the down projection uses the dequantized a. Returns Y [n][H] float64 (and
    the SwiGLU output's codes and scales with ``return_act``)."""
    Wg, Wu, Wd = expert.values()
    xc, xs = quantize(np.asarray(X, dtype=np.float32), g_in)
    Xq = dequantize(xc, xs, g_in)
    a = (silu(Xq @ Wg.T) * (Xq @ Wu.T)).astype(np.float32)
    ac, as_ = quantize(a, g_act)
    Y = dequantize(ac, as_, g_act) @ Wd.T
    return (Y, ac, as_) if return_act else Y
