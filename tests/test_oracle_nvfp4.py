"""Pins for the oracle's NVFP4 formats and experts (E2M1 values, E4M3 block
scales, FP32 scales): decoded values against the format definition and
PyTorch's float8_e4m3fn, roundings against an arithmetic construction, block
quantization against exact round trips and closed forms, and the NVFP4 FFN
against the bf16 oracle FFN."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4 as q
from oracle.experts import swiglu_ffn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_values_and_rounding_match_the_worked_table():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_e2m1.json")))
    v = q.e2m1_decode(np.array(g["codes"]))
    assert np.array_equal(v, np.array(g["values"]))
    assert np.array_equal(np.signbit(v), np.signbit(np.array(g["values"])))
    r = g["round_to_nearest_even"]
    assert q.e2m1_round(np.array(r["inputs"])).tolist() == r["codes"]


def test_e4m3_decode_matches_torch_on_all_256_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = q.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2
    assert np.array_equal(mine[~nan], ref[~nan])
    assert q.e4m3_decode(np.array([0x7E]))[0] == 448.0 and q.e4m3_decode(np.array([1]))[0] == 2.0 ** -9


def test_e4m3_round_matches_torch():
    # every midpoint between neighbouring finite values, the values themselves,
    # and random FP32 values, up to 464 (torch gives NaN from 480 on; the
    # reading here saturates, see below)
    mags = q.e4m3_decode(np.arange(0x7F))
    mids = (mags[:-1] + mags[1:]) / 2
    rng = np.random.default_rng(3)
    rand = np.exp(rng.uniform(np.log(1e-4), np.log(464.0), 20000))
    v = np.concatenate([mags, mids, rand, [464.0]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q.e4m3_round(v.astype(np.float64)), ref)
    # saturating reading: beyond the largest finite value the scale is 448
    assert q.e4m3_round(np.array([465.0, 480.0, 1e6])).tolist() == [0x7E] * 3


def test_e2m1_round_matches_an_arithmetic_construction():
    # Independent construction: magnitudes >= 1 keep two significant bits
    # (scale by the exponent, np.rint half-to-even, scale back), magnitudes
    # below 1 round to a multiple of 0.5, and the result saturates at 6.
    rng = np.random.default_rng(4)
    mags = q.e2m1_decode(np.arange(8))
    mids = (mags[:-1] + mags[1:]) / 2
    v = np.concatenate([mags, mids, rng.uniform(0, 8, 20000), rng.uniform(0, 1, 5000)])
    v = np.concatenate([v, -v]).astype(np.float32).astype(np.float64)
    a = np.abs(v)
    ex = np.floor(np.log2(np.maximum(a, 1.0)))
    r = np.where(a >= 1.0, np.ldexp(np.rint(np.ldexp(a, -(ex - 1).astype(int))), (ex - 1).astype(int)),
                 np.rint(a * 2) / 2)
    r = np.minimum(r, 6.0)
    got = q.e2m1_decode(q.e2m1_round(v))
    assert np.array_equal(np.abs(got), r)
    assert np.array_equal(np.signbit(got), np.signbit(v))


def test_representable_blocks_round_trip_exactly():
    # x = q * s * g with a power-of-two g and a code of magnitude 6 in every
    # block: amax / (6 g) = s exactly and x / (s g) = q exactly, so the
    # quantizer must return the very codes and scales (any wrong grouping,
    # order of operations or scale formula breaks this).
    rng = np.random.default_rng(5)
    rows, K, g = 12, 96, 2.0 ** -6
    codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    blocks = codes.reshape(rows, K // 16, 16)
    pos = rng.integers(0, 16, (rows, K // 16))
    np.put_along_axis(blocks, pos[..., None], np.where(rng.random((rows, K // 16, 1)) < 0.5, 7, 15), axis=2)
    scales = rng.integers(0x08, 0x7F, (rows, K // 16)).astype(np.uint8)   # normal E4M3 scales
    x = q.dequantize(codes, scales, g)
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)  # exact in FP32
    c2, s2 = q.quantize(x, g)
    assert np.array_equal(s2, scales)
    # +-0 codes may come back as the other zero only where the value is 0
    assert np.array_equal(np.where(q.e2m1_decode(codes) == 0, 0, codes), np.where(q.e2m1_decode(c2) == 0, 0, c2))


def test_each_block_of_16_has_its_own_scale_and_zero_blocks_code_zero():
    g = 1.0
    row = np.concatenate([np.full(16, 0.012), np.full(16, 1.0), np.full(16, 96.0), np.zeros(16)])[None]
    codes, scales = q.quantize(row, g)
    expect = q.e4m3_round(np.array([0.012, 1.0, 96.0, 0.0]) / 6.0)
    assert scales[0].tolist() == expect.tolist()
    assert scales[0, 3] == 0 and np.all(codes[0, 48:] == 0)
    # a constant block quantizes to the largest code (amax maps to 6)
    assert np.all(codes[0, 16:32] == 7) and np.all(codes[0, 32:48] == 7)


def test_sign_symmetry_and_error_bound():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((20, 256)) * np.exp(rng.uniform(-4, 4, (20, 1)))).astype(np.float32)
    g = 2.0 ** -6
    c, s = q.quantize(x, g)
    cn, sn = q.quantize(-x, g)
    assert np.array_equal(s, sn) and np.array_equal(cn, c ^ 8)
    xq = q.dequantize(c, s, g)
    step = np.repeat(q.e4m3_decode(s), 16, axis=1) * g     # one code unit of each block
    # |x - x~| is at most one E2M1 spacing unit (1 between 4 and 6) plus what
    # saturation at 6 clips
    excess = np.maximum(np.abs(x) - 6 * step, 0)
    assert np.all(np.abs(x - xq) <= step * 1.0 + excess + 1e-30)
    assert np.mean(np.abs(x - xq) / np.abs(x).max(axis=1, keepdims=True)) < 0.05


def test_expert_scale_puts_the_largest_weight_on_scale_448():
    rng = np.random.default_rng(7)
    Wg, Wu = rng.standard_normal((2, 32, 64)).astype(np.float32) * 0.02
    Wd = rng.standard_normal((64, 32)).astype(np.float32) * 0.02
    Wd[5, 17] = 0.3                                  # the expert's largest |w|
    e = q.Nvfp4Expert(Wg, Wu, Wd)
    assert e.g == np.float32(0.3) / np.float32(2688.0)
    assert e.down[1][5, 1] == 0x7E                   # its block's scale is 448
    assert e.down[0][5, 17] == 7                     # and its code 6
    assert e.gate[1].max() < 0x7E


def test_pack_puts_element_zero_in_the_low_nibble():
    codes = np.array([[1, 2, 3, 4, 15, 0]], dtype=np.uint8)
    p = q.pack_codes(codes)
    assert p.tolist() == [[0x21, 0x43, 0x0F]]
    assert np.array_equal(q.unpack_codes(p), codes)


def _representable(rng, shape, g, top=False):
    codes = rng.integers(0, 16, shape).astype(np.uint8)
    blocks = codes.reshape(shape[0], shape[1] // 16, 16)
    blocks[..., 0] = 7                                # every block reaches 6
    scales = rng.integers(0x20, 0x40, (shape[0], shape[1] // 16)).astype(np.uint8)
    if top:
        scales[0, 0] = 0x7E                           # one block at scale 448: amax = 6 * 448 * g
    return q.dequantize(codes, scales, g)


def test_ffn_with_representable_operands_matches_the_bf16_ffn_up_to_the_act_quantization():
    rng = np.random.default_rng(8)
    H, F, n = 64, 32, 5
    g_w = 2.0 ** -14
    Wg, Wu = _representable(rng, (F, H), g_w), _representable(rng, (F, H), g_w)
    Wd = _representable(rng, (H, F), g_w, top=True)
    e = q.Nvfp4Expert(Wg, Wu, Wd)
    assert e.g == np.float32(g_w)
    for (c, s), W in zip((e.gate, e.up, e.down), (Wg, Wu, Wd)):
        assert np.array_equal(q.dequantize(c, s, e.g), W)
    X = _representable(rng, (n, H), 2.0 ** -6)
    a = (X @ Wg.T) / (1 + np.exp(-(X @ Wg.T))) * (X @ Wu.T)
    g_act = 2.0 ** np.floor(np.log2(np.abs(a).max() / 2688))   # the SwiGLU output's FP32 scale
    Y, ac, as_ = q.ffn(X, e, 2.0 ** -6, g_act, return_act=True)
    assert np.all(as_ > 0)
    ref = swiglu_ffn(X, Wg, Wu, Wd)
    # the only rounding left is the act quantization: |dY| <= sum_f |Wd| * |a - a~|
    da = np.abs(a - q.dequantize(ac, as_, g_act))
    bound = da @ np.abs(Wd).T                         # [n][H]
    assert np.all(np.abs(Y - ref) <= bound * (1 + 1e-9) + 1e-15)
    assert np.abs(Y - ref).max() > 0                  # the act quantization is really applied
    assert np.abs(Y).max() > 0
    # doubling every weight doubles the expert's FP32 scale and leaves codes and block scales alone
    e2 = q.Nvfp4Expert(2 * Wg, 2 * Wu, 2 * Wd)
    assert e2.g == 2 * e.g
    for a, b in zip((e.gate, e.up, e.down), (e2.gate, e2.up, e2.down)):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
