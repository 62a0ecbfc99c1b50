"""Pins for the oracle's rounding primitives.

RN16 is checked against two things the oracle does not use: torch's fp32 ->
bf16 conversion (a library routine, round to nearest even) for random fp32 bit
patterns, and exact rational rounding for doubles, ties and the edges of the
format (subnormals, overflow threshold).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from _exact import rn16_bits, rn16_of_rn32_bits, is_nan_bits


def test_fp_env_keeps_subnormals(oracle_lib):
    assert oracle_lib.dto_fp_env_ok() == 1


def test_rn16_matches_torch_cast_on_random_fp32_bits(oracle_lib):
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2**32, size=60000, dtype=np.uint64).astype(np.uint32)
    # add specials and the neighbourhood of the bf16 rounding boundary
    extra = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0x00000001,
                      0x00008000, 0x00018000, 0x3F808000, 0x3F818000, 0x3F807FFF,
                      0x7F7F7FFF, 0x7F7F8000, 0x7F7FFFFF, 0x007F8000, 0x00800000],
                     dtype=np.uint32)
    bits = np.concatenate([bits, extra])
    f32 = bits.view(np.float32)
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rn16 = oracle_lib.dto_rn16
    got = np.array([rn16(float(v)) for v in f32], dtype=np.uint16)
    nan = np.isnan(f32)
    assert np.all(got[~nan] == ref[~nan])
    assert all(is_nan_bits(int(b)) for b in got[nan])


def test_rn16_exact_rational_rounding_of_doubles(oracle_lib):
    rng = np.random.default_rng(99)
    vals = []
    # random doubles spanning the bf16 range, including the subnormal range
    for e in rng.integers(-140, 128, size=3000):
        vals.append(float(rng.uniform(1, 2)) * 2.0 ** int(e) * (1 if rng.random() < .5 else -1))
    # exact ties and near-ties on the bf16 grid
    for k in range(128, 256, 7):
        for E in (-133, -126, -1, 0, 5, 127):
            mid = (k + 0.5) * 2.0 ** (E - 7)
            vals += [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), -mid]
    # overflow threshold (2 - 2^-8) * 2^127 and its neighbours
    thr = (2 - 2**-8) * 2.0 ** 127
    vals += [thr, np.nextafter(thr, 0), -thr, 2.0 ** -134, 2.0 ** -134 * (1 + 2**-40),
             2.0 ** -135, 3 * 2.0 ** -135]
    for v in vals:
        assert oracle_lib.dto_rn16(v) == rn16_bits(Fraction(v)), v


def test_rn16_of_rn32_double_rounding(oracle_lib):
    # 1 + 2^-8 + 2^-30: RN32 drops the 2^-30 and lands on the bf16 midpoint,
    # which ties to even (1.0); a single rounding would go up.
    v = 1 + 2**-8 + 2**-30
    assert oracle_lib.dto_rn16_of_rn32(v) == 0x3F80 == rn16_of_rn32_bits(Fraction(v))
    assert oracle_lib.dto_rn16(v) == 0x3F81 == rn16_bits(Fraction(v))
    rng = np.random.default_rng(5)
    for _ in range(2000):
        v = float(rng.standard_normal()) * 2.0 ** int(rng.integers(-130, 100))
        assert oracle_lib.dto_rn16_of_rn32(v) == rn16_of_rn32_bits(Fraction(v))


def test_bf16_roundtrip_all_patterns(oracle_lib):
    # every finite bf16 value is a fixed point of RN16
    f = oracle_lib.dto_bf16_to_double
    r = oracle_lib.dto_rn16
    for b in range(0, 1 << 16, 3):
        v = f(b)
        if np.isnan(v):
            continue
        assert r(v) == b
