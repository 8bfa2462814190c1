"""Pins for the oracle's bf16 conversions (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import bf16_bits_to_f64, f64_to_bf16_bits, round_bf16


def test_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x7F7F], np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, np.inf, -np.inf, 2.0 ** -133, float.fromhex("0x1.fep127")]
    got = bf16_bits_to_f64(bits)
    assert got.tolist() == want
    assert np.signbit(got[3])


def test_rounding_matches_torch_for_float32_inputs():
    # torch's float32 -> bfloat16 cast rounds to nearest even; for inputs that
    # are float32 values the oracle's direct rounding must agree bit for bit.
    g = np.random.default_rng(1)
    x = np.concatenate([
        g.standard_normal(200000).astype(np.float32),
        (g.standard_normal(20000) * 1e30).astype(np.float32),
        (g.standard_normal(20000) * 1e-38).astype(np.float32),   # subnormal range
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_ties_go_to_even():
    one = 1.0
    assert round_bf16(np.array([one + 2.0 ** -8]))[0] == 1.0                   # tie, 1.0 is even
    assert round_bf16(np.array([one + 3 * 2.0 ** -8]))[0] == one + 2.0 ** -6   # tie, round up to even
    assert round_bf16(np.array([-(one + 2.0 ** -8)]))[0] == -1.0


def test_direct_rounding_from_float64_has_no_double_rounding():
    # 1 + 2^-8 + 2^-30 lies just above the tie: correct rounding goes up, while
    # rounding through float32 first would land on the tie and go down to 1.0.
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30])
    assert round_bf16(x)[0] == 1.0 + 2.0 ** -7


def test_overflow_and_nan():
    x = np.array([float.fromhex("0x1.ffp127"), np.nan, -np.inf])
    y = round_bf16(x)
    assert y[0] == np.inf and np.isnan(y[1]) and y[2] == -np.inf
    assert f64_to_bf16_bits(np.array([np.nan]))[0] == 0x7FC0
