"""Pins for the oracle's rotate-half RoPE.

Source: ERNIE-Image fusion page, section 2: round(round(x1*cos1) +
round(-x2*sin1)) per element, the eager chunk/neg/cat/mul/add chain, tail
columns passed through.  Pins: hand-worked examples (golden file), the zero
angle, fp64 invariants of a rotation (pair norm, relative position), tail
passthrough, and the eager chain itself run by torch on the CPU in bf16.
"""
import numpy as np
import pytest
import torch

from fractions import Fraction

import oracle
from _exact import rn16_bits
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _golden import load


def _tables(freqs):
    return oracle.rope_cos_sin(freqs)


def test_hand_examples():
    for (vals, out) in load("rope_rotate_half_hand.txt"):
        x0, x1, c0, c1, s0, s1 = vals
        x = np.array([x0, x1], np.uint16).reshape(1, 1, 1, 2)
        cos = np.array([[c0, c1]], np.uint16)
        sin = np.array([[s0, s1]], np.uint16)
        got = oracle.rope_rotate_half(x, cos, sin)
        assert got.reshape(-1).tolist() == out


def test_zero_angle_returns_x():
    x = W.normal_bf16((1, 8, 3, 32), 11, 0)
    xb = oracle.bf16_bits(x)
    rot = 24
    cos = np.full((8, rot), 0x3F80, np.uint16)
    sin = np.zeros((8, rot), np.uint16)
    out = oracle.rope_rotate_half(xb, cos, sin)
    # numerically equal (the sign of a zero may change: -0 + +0 = +0)
    assert np.array_equal(oracle.bits_to_f64(out), oracle.bits_to_f64(xb))


def test_tail_columns_pass_through_bitwise():
    x = W.normal_bf16((2, 5, 3, 40), 12, 0)
    xb = oracle.bf16_bits(x)
    rng = np.random.default_rng(0)
    rot = 24
    cos = oracle.rn16_array(rng.uniform(-1, 1, (10, rot)))
    sin = oracle.rn16_array(rng.uniform(-1, 1, (10, rot)))
    out = oracle.rope_rotate_half(xb, cos, sin)
    assert np.array_equal(out[..., rot:], xb[..., rot:])


def test_fp64_rotation_preserves_pair_norms():
    rng = np.random.default_rng(1)
    B, S, H, D, rot = 1, 16, 2, 32, 24
    freqs = W.freqs_1d(S, B, rot).numpy().astype(np.float64) * 1.7
    cos, sin = oracle.rope_cos_sin_f64(freqs)
    x = rng.standard_normal((B, S, H, D))
    out = oracle.rope_rotate_half_f64(x, cos, sin)
    h = rot // 2
    n_in = x[..., :h] ** 2 + x[..., h:rot] ** 2
    n_out = out[..., :h] ** 2 + out[..., h:rot] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-13, atol=1e-13)
    assert np.array_equal(out[..., rot:], x[..., rot:])


def test_fp64_dot_product_depends_on_position_difference():
    rng = np.random.default_rng(2)
    D, rot = 16, 16
    q = rng.standard_normal((1, 1, 1, D))
    k = rng.standard_normal((1, 1, 1, D))

    inv = 10000.0 ** (-2.0 * np.arange(rot // 2) / rot)

    def rope_at(v, pos):
        half = pos * inv  # angles in double, laid out cat(half, half)
        f = np.concatenate([half, half])
        c, s = oracle.rope_cos_sin_f64(f.reshape(1, 1, 1, rot))
        return oracle.rope_rotate_half_f64(v, c, s).reshape(-1)

    for m, n, shift in [(3, 1, 5), (10, 4, 17), (0, 7, 100)]:
        a = rope_at(q, m) @ rope_at(k, n)
        b = rope_at(q, m + shift) @ rope_at(k, n + shift)
        assert abs(a - b) < 1e-12 * max(1.0, abs(a))
    # and it does change with the difference
    assert abs(rope_at(q, 3) @ rope_at(k, 1) - rope_at(q, 3) @ rope_at(k, 2)) > 1e-6


def _eager_chain(x, cos, sin):
    """The eager bf16 chain of the pages, run by torch on the CPU."""
    B, S, H, D = x.shape
    rot = cos.shape[-1]
    c = cos.view(B, S, 1, rot)
    s = sin.view(B, S, 1, rot)
    x_rot, tail = x[..., :rot], x[..., rot:]
    x1, x2 = x_rot.chunk(2, dim=-1)
    rotated = torch.cat((-x2, x1), dim=-1)
    y = x_rot * c + rotated * s
    return torch.cat((y, tail), dim=-1)


@pytest.mark.parametrize("name", ["tiny", "image"])
def test_matches_torch_cpu_eager_chain(name):
    wl = W.WORKLOADS[name]
    S = min(wl.S, 512)
    x = W.rope_inputs(wl, "q")[:, :S]
    freqs = W.freqs_for(wl)[:S]
    cos, sin = _tables(freqs.numpy())
    out = oracle.rope_rotate_half(oracle.bf16_bits(x), cos, sin)
    ref = _eager_chain(x, oracle.from_bits(cos), oracle.from_bits(sin))
    assert np.array_equal(out, oracle.bf16_bits(ref))


def test_matches_eager_chain_with_unrelated_halves_and_strides():
    # tables whose two halves differ catch a swapped or shifted column index;
    # x is a strided view of a fused (B, S, 3H, D) buffer
    rng = np.random.default_rng(3)
    B, S, H, D, rot = 2, 7, 3, 24, 16
    qkv = W.normal_bf16((B, S, 3 * H, D), 21, 0)
    x = qkv[:, :, H:2 * H]
    cos = oracle.rn16_array(rng.uniform(-2, 2, (B * S, rot)))
    sin = oracle.rn16_array(rng.uniform(-2, 2, (B * S, rot)))
    xb = oracle.bf16_bits(qkv)[:, :, H:2 * H]
    out = oracle.rope_rotate_half(xb, cos, sin)
    ref = _eager_chain(x.contiguous(), oracle.from_bits(cos), oracle.from_bits(sin))
    assert np.array_equal(out, oracle.bf16_bits(ref))


def test_exhaustive_x_against_eager_chain():
    # every bf16 x (as x0, with a fixed partner) against a few (c, s) pairs whose
    # products are multiples of 2^-149, hence exact in fp32, so torch's fp32
    # multiply followed by a bf16 cast is one rounding of the exact product
    allx = np.arange(1 << 16, dtype=np.uint16)
    partner = np.full_like(allx, 0x3FA0)  # 1.25
    x = np.stack([allx, partner], axis=-1).reshape(1, -1, 1, 2)
    S = x.shape[1]
    for c, s in [(0x3F80, 0x0000), (0x3F35, 0x3F35), (0xBE9A, 0x3F74), (0x3C23, 0xBF7F)]:
        cos = np.full((S, 2), c, np.uint16)
        sin = np.full((S, 2), s, np.uint16)
        out = oracle.rope_rotate_half(x, cos, sin)
        ref = oracle.bf16_bits(_eager_chain(oracle.from_bits(x), oracle.from_bits(cos),
                                            oracle.from_bits(sin)))
        o, r = oracle.bits_to_f64(out), oracle.bits_to_f64(ref)
        same = (out == ref) | (np.isnan(o) & np.isnan(r))
        assert same.all()


def test_tiny_products_round_like_the_fp32_chain():
    # A product of two bf16 values has a 16-bit significand, so it is exact in
    # fp32 unless it lies below 2^-134, where both roundings give 0 or the
    # nearest subnormal the same way: rounding the exact product once (the
    # oracle) equals the eager chain's fp32 multiply and bf16 cast.  Sampled on
    # products near and below the bf16 subnormal range.
    from _exact import rn16_of_rn32_bits
    rng = np.random.default_rng(4)
    mx = rng.integers(128, 256, 3000)
    mc = rng.integers(128, 256, 3000)
    esum = rng.integers(-141, -128, 3000)
    for a, b, e in zip(mx, mc, esum):
        ex = int(e) // 2
        ec = int(e) - ex
        x0 = float(a) * 2.0 ** (ex - 7)
        c0 = float(b) * 2.0 ** (ec - 7)
        xb, cb = oracle.rn16(x0), oracle.rn16(c0)
        x = np.array([xb, 0], np.uint16).reshape(1, 1, 1, 2)
        cos = np.array([[cb, cb]], np.uint16)
        sin = np.zeros((1, 2), np.uint16)
        got = int(oracle.rope_rotate_half(x, cos, sin).reshape(-1)[0])
        prod = Fraction(oracle.bits_to_f64(np.array([xb], np.uint16))[0]) * \
            Fraction(oracle.bits_to_f64(np.array([cb], np.uint16))[0])
        assert got == rn16_bits(prod) == rn16_of_rn32_bits(prod)
