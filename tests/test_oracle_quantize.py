"""Pins of the oracle quantizer: hand-derived cases, brute force in exact
rational arithmetic, and bounds that hold for any input."""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle.quantize import quantize_block, block_scale, dequantize

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_cases.txt")


def _golden_cases():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tag, *vals = line.split()
            if tag == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif tag == "x":
                cur["x"] = np.array([float(v) for v in vals], dtype=np.float32)
            elif tag == "scale":
                cur["scale"] = np.float32(float(vals[0]))
            elif tag == "q":
                cur["q"] = np.array([int(v) for v in vals], dtype=np.int8)
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_cases(case):
    q, s = quantize_block(case["x"])
    assert s.dtype == np.float32 and s == case["scale"]
    assert np.array_equal(q, case["q"])


# -- an independent brute force in exact rational arithmetic ----------------

def _round_half_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def _to_f32(fr: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value (ties to even), normal range."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (e - 23)
    return sign * _round_half_even(a / quantum) * quantum


def _brute_quantize(xs):
    xs = [Fraction(float(v)) for v in xs]
    m = max(abs(v) for v in xs)
    s = Fraction(1) if m < Fraction(float(np.float32(1e-6))) else _to_f32(m / 127)
    q = []
    for v in xs:
        r = _to_f32(v / s) if v != 0 else Fraction(0)
        q.append(max(-127, min(127, _round_half_even(r))))
    return q, s


def _bf16_block(gen, n, scale):
    return (torch.randn(n, generator=gen) * scale).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_random_blocks(seed):
    gen = torch.Generator().manual_seed(seed)
    scale = [1e-3, 0.1, 1.0, 3.7, 250.0][seed % 5]
    x = _bf16_block(gen, 64, scale)
    if seed % 7 == 3:  # force exact quotient ties: x = (k + 1/2) * s with s a power of two
        x = np.array([(k + 0.5) * 0.25 for k in range(-60, 60)] + [127 * 0.25], dtype=np.float32)
    q, s = quantize_block(x)
    bq, bs = _brute_quantize(x)
    assert Fraction(float(s)) == bs
    assert q.tolist() == bq


def test_reciprocal_variant_differs_somewhere():
    """The page multiplies by 1/scale and rounds ties away from zero; the
    reading here divides and rounds ties to even. Show the two are different
    functions on bf16 inputs, so that the tests above do pin the choice."""
    x = np.array([127.0, 2.5, -0.5, 1.5], dtype=np.float32)
    q, _ = quantize_block(x)
    away = np.sign(x) * np.floor(np.abs(x) + 0.5)
    assert not np.array_equal(q, away.astype(np.int8))


def test_guard_reading_agrees_on_all_bf16_inputs():
    # "max < 1e-6 -> 1.0" and "max > 1e-6 -> max/127" differ only at max == fp32(1e-6),
    # which no bf16 value equals.
    all_bf16 = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = all_bf16.float().abs().numpy()
    assert not np.any(vals == np.float32(1e-6))


def test_bounds_on_random_data():
    gen = torch.Generator().manual_seed(11)
    for trial in range(50):
        x = _bf16_block(gen, 16 * 64, 2.0 ** (trial % 9 - 4))
        q, s = quantize_block(x)
        assert q.min() >= -127 and q.max() <= 127
        m = np.abs(x).max()
        # the largest magnitude maps to +-127
        assert np.abs(q.astype(np.int32)).max() == 127
        assert np.isclose(float(s) * 127, m, rtol=1e-6)
        err = np.abs(dequantize(q, s) - x.astype(np.float64))
        # |q*s - x| <= s/2, widened by the fp32 rounding of x/s (|x/s| <= 127.5,
        # so one ulp of the quotient is at most 2^-17) and of s itself.
        assert err.max() <= float(s) * (0.5 + 2.0 ** -16)


def test_scale_is_fp32_division():
    x = np.array([0.0, -1.0, 0.5, 2.0], dtype=np.float32)
    assert block_scale(x) == np.float32(2.0) / np.float32(127.0)
