"""Pins for the oracle's fp16 / bf16 rounding (round to nearest, ties to even)."""

from fractions import Fraction

import numpy as np
import torch

from oracle import numerics


def _f16_value(bits):
    return Fraction(float(np.uint16(bits).view(np.float16)))


def test_f16_all_midpoints_round_to_even():
    # every pair of adjacent positive finite fp16 values: the exact midpoint
    # must round to the neighbour with the even significand
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    hi = lo + np.uint16(1)
    vlo = lo.view(np.float16).astype(np.float64)
    vhi = hi.view(np.float16).astype(np.float64)
    mid = (vlo + vhi) / 2  # exact in fp64
    got = numerics.to_f16(mid).view(np.uint16)
    want = np.where(lo % 2 == 0, lo, hi)
    assert np.array_equal(got, want)
    # just above / below the midpoint goes to the nearer neighbour
    up = numerics.to_f16(np.nextafter(mid, np.inf)).view(np.uint16)
    dn = numerics.to_f16(np.nextafter(mid, -np.inf)).view(np.uint16)
    assert np.array_equal(up, hi)
    assert np.array_equal(dn, lo)


def test_f16_single_rounding_from_double():
    # a value a hair above an fp16 midpoint but within float32's rounding of it:
    # rounding through float32 first would land on the midpoint and then go to
    # even; one rounding from the double must go up.
    lo = np.uint16(0x3C00)  # 1.0, even significand
    hi = np.uint16(0x3C01)
    m = (float(lo.view(np.float16)) + float(hi.view(np.float16))) / 2
    x = m + 2.0 ** -40
    assert np.float32(x) == np.float32(m)  # float32 cannot see the difference
    assert numerics.to_f16(x).view(np.uint16) == hi


def test_f16_exact_rational_rounding_random():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(2000) * 10.0 ** rng.uniform(-6, 4, 2000)
    got = numerics.to_f16(x).view(np.uint16)
    for xi, gi in zip(x, got):
        v = Fraction(float(xi))
        cand = [int(gi) - 1, int(gi), int(gi) + 1] if xi > 0 else None
        if xi <= 0:
            continue
        dists = [(abs(_f16_value(c) - v), c % 2, c) for c in cand if 0 <= c < 0x7C00]
        best = min(dists)
        assert best[2] == int(gi)


def test_f16_overflow_boundary():
    assert np.isinf(numerics.to_f16(65520.0))  # tie between 65504 (odd) and inf
    assert numerics.to_f16(65519.99) == np.float16(65504.0)


def test_bf16_matches_torch_conversion():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(200_000) * 10.0 ** rng.uniform(-30, 30, 200_000)).astype(np.float32)
    # include exact ties and their neighbours
    ties = ((rng.integers(0, 0x7F00, 5000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.nextafter(ties, np.float32(np.inf))])
    got = numerics.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_ties_go_to_even_exactly():
    hi = np.arange(0x3F00, 0x4100, dtype=np.uint32)
    x = ((hi << 16) | 0x8000).view(np.float32)
    got = numerics.f32_to_bf16_bits(x).astype(np.uint32)
    want = np.where(hi % 2 == 0, hi, hi + 1)
    assert np.array_equal(got, want)
    # and the chosen neighbour is at exactly half an ulp (a true tie)
    lo_v = (hi << 16).view(np.float32)
    hi_v = ((hi + 1) << 16).view(np.float32)
    for v, a, b in zip(x[:16], lo_v[:16], hi_v[:16]):
        assert Fraction(float(v)) - Fraction(float(a)) == Fraction(float(b)) - Fraction(float(v))


def test_bf16_roundtrip_values():
    b = np.arange(0, 0x7F80, 97, dtype=np.uint16)
    v = numerics.bf16_bits_to_f64(b)
    assert np.array_equal(numerics.f32_to_bf16_bits(v.astype(np.float32)), b)
