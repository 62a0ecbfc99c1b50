"""Pins for the oracle's RMSNorm fused with the residual add.

Source: the sequence-parallelism post, per-token normalisation and residual
add, Pre-Norm layer order.  Pins: unit RMS in fp64 before the weight, row
subsets equal the rows of the full run (per-token independence), constant rows
and C = 1 against exact arithmetic, the hand-worked golden file, and torch's
CPU F.rms_norm within the stated tolerance.
"""
import math
from fractions import Fraction

import mpmath
import numpy as np
import torch
import torch.nn.functional as Fn

import oracle
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _exact import rn16_bits, bf16_value
from _golden import load

EPS = float(np.float32(1e-6))


def test_hand_examples():
    rows = load("rmsnorm_residual_hand.txt")
    x = np.array([r[0][:4] for r in rows], np.uint16)
    res = np.array([r[0][4:] for r in rows], np.uint16)
    w = oracle.rn16_array(np.array([1, 2, 0.5, -1.0]))
    h, y = oracle.rmsnorm_residual(x, res, w, EPS)
    assert h.tolist() == [r[1] for r in rows]
    assert y.tolist() == [r[2] for r in rows]


def test_fp64_unit_rms_before_weight():
    rng = np.random.default_rng(0)
    T, C = 7, 96
    x = rng.standard_normal((T, C))
    r = rng.standard_normal((T, C)) * 2
    h, y = oracle.rmsnorm_residual_f64(x, r, np.ones(C), EPS)
    assert np.allclose(h, x + r, rtol=0, atol=0)
    ms = (h ** 2).mean(axis=1)
    rms_y = np.sqrt((y ** 2).mean(axis=1))
    assert np.allclose(rms_y, np.sqrt(ms / (ms + EPS)), rtol=1e-14)
    # the weight scales features after normalisation
    w = rng.standard_normal(C)
    _, yw = oracle.rmsnorm_residual_f64(x, r, w, EPS)
    assert np.allclose(yw, y * w[None, :], rtol=1e-14, atol=1e-300)


def test_row_subsets_equal_rows_of_full_run():
    x, r, w = W.rmsnorm_inputs(W.WORKLOADS["tiny"])
    xb, rb, wb = (oracle.bf16_bits(t) for t in (x, r, w))
    h, y = oracle.rmsnorm_residual(xb, rb, wb, EPS)
    for a, b in [(0, 1), (3, 17), (100, 256), (255, 256)]:
        hs, ys = oracle.rmsnorm_residual(xb[a:b], rb[a:b], wb, EPS)
        assert np.array_equal(hs, h[a:b]) and np.array_equal(ys, y[a:b])


def test_constant_row_and_single_feature():
    mpmath.mp.dps = 60
    for a_bits, w_bits, C in [(0x3FC0, 0x3F80, 8), (0xC0A0, 0x3F40, 5), (0x3A80, 0xBF90, 1),
                              (0x0001, 0x3F80, 3)]:
        a, wv = bf16_value(a_bits), bf16_value(w_bits)
        x = np.full((1, C), a_bits, np.uint16)
        res = np.zeros((1, C), np.uint16)
        w = np.full(C, w_bits, np.uint16)
        h, y = oracle.rmsnorm_residual(x, res, w, EPS)
        # y = w * a / sqrt(a^2 + eps), rounded once
        ex = mpmath.mpf(wv) * mpmath.mpf(a) / mpmath.sqrt(mpmath.mpf(a) ** 2 + mpmath.mpf(EPS))
        assert np.all(h == a_bits)
        assert np.all(y == rn16_bits(ex)), (hex(a_bits), hex(int(y[0, 0])), hex(rn16_bits(ex)))


def test_residual_is_bf16_sum():
    x, r, w = W.rmsnorm_inputs(W.WORKLOADS["tiny"])
    h, _ = oracle.rmsnorm_residual(*(oracle.bf16_bits(t) for t in (x, r, w)), EPS)
    assert np.array_equal(h, oracle.bf16_bits(x + r))


def _ulp_diff(a, b):
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, 0x8000 - (u & 0x7FFF), 0x8000 + u)
    return np.abs(key(a) - key(b))


def test_against_torch_cpu_rms_norm_within_tolerance():
    x, r, w = W.rmsnorm_inputs(W.WORKLOADS["tiny"])
    h = x + r
    ref = Fn.rms_norm(h.double(), (h.shape[1],), w.double(), EPS).to(torch.bfloat16)
    _, y = oracle.rmsnorm_residual(*(oracle.bf16_bits(t) for t in (x, r, w)), EPS)
    d = _ulp_diff(y, oracle.bf16_bits(ref))
    assert d.max() <= 1
    assert np.count_nonzero(d) <= 1e-4 * d.size + 1
