"""Pins for the oracle's bfloat16 codec (IEEE 754 round to nearest even)."""
import numpy as np
import torch

from oracle import bf16


def _torch_bits(v32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_matches_library_cast_on_float32_inputs():
    # For inputs that are exactly float32 there is no double-rounding hazard,
    # so PyTorch's float32 -> bfloat16 cast (round to nearest even) is a
    # reference for the direct float64 rounding.
    rng = np.random.default_rng(1)
    v = rng.standard_normal(200000).astype(np.float32)
    v *= np.exp2(rng.integers(-140, 128, v.size)).astype(np.float32)
    v = v[np.isfinite(v)]
    assert np.array_equal(bf16.encode(v.astype(np.float64)), _torch_bits(v))


def test_ties_go_to_even():
    one = 1.0
    assert bf16.round_bf16(one + 2.0 ** -8) == 1.0                     # tie, 1.0 is even
    assert bf16.round_bf16(one + 3 * 2.0 ** -8) == one + 2.0 ** -6     # tie, round up to even
    assert bf16.round_bf16(-(one + 2.0 ** -8)) == -1.0


def test_direct_rounding_avoids_double_rounding():
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30      # just above a tie
    assert bf16.round_bf16(v) == 1.0 + 2.0 ** -7
    # going through float32 first lands exactly on the tie and rounds down
    via32 = _torch_bits(np.array([v], dtype=np.float32))
    assert bf16.decode(via32)[0] == 1.0


def test_overflow_and_specials():
    mx = bf16.BF16_MAX
    assert bf16.round_bf16(mx) == mx
    assert bf16.round_bf16(mx + 2.0 ** 119) == np.inf          # exactly half an ulp above: tie -> inf (even)
    assert bf16.round_bf16(mx + 2.0 ** 118) == mx
    assert bf16.round_bf16(-2.0 ** 128) == -np.inf
    assert np.isnan(bf16.round_bf16(np.nan))
    assert bf16.round_bf16(np.inf) == np.inf
    z = bf16.round_bf16(-0.0)
    assert z == 0.0 and np.signbit(z)


def test_subnormals():
    assert bf16.round_bf16(2.0 ** -133) == 2.0 ** -133
    assert bf16.round_bf16(2.0 ** -134) == 0.0                  # tie between 0 and 2^-133 -> 0
    assert bf16.round_bf16(3 * 2.0 ** -134) == 2.0 ** -132      # tie between 1 and 2 units -> 2
    assert bf16.round_bf16(2.0 ** -126 - 2.0 ** -140) == 2.0 ** -126


def test_every_bit_pattern_round_trips():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = bf16.decode(bits)
    fin = ~np.isnan(v)
    assert np.array_equal(bf16.encode(v[fin]), bits[fin])


def test_ulp_distance():
    a = bf16.encode(np.array([1.0, 1.0, -1.0, 0.0]))
    b = bf16.encode(np.array([1.0 + 2 ** -7, 1.0 + 2 ** -6, 1.0, -0.0]))
    assert bf16.ulp_distance(a, b).tolist() == [1, 2, 2 * 0x3F80, 0]
