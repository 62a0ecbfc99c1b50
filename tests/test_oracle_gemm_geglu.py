"""Pins for the oracle of GEGLU after the gate_up projection.

gate_up_bf16 is the projection x W^T rounded once to bf16; gemm_gelu_and_mul
feeds it to the pinned GEGLU.  Checked against hand-worked rows, against exact
rational sums, against the GEGLU oracle when the weights are identities, and
the fp32-accumulation bounds against simulated fp32 sums in shuffled orders.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
from _exact import round_fraction
from _golden import load
from diffusion_transformer_elementwise_rotate_b300 import workloads as W

bits = oracle.bf16_bits


def _val(b):
    return float(oracle.bits_to_f64(np.array([b], np.uint16))[0])


def test_hand_worked_rows():
    for xrow, grow, urow, (out,) in load("gemm_gelu_and_mul_hand.txt"):
        x = np.array([xrow], np.uint16)
        w = np.array([grow, urow], np.uint16)
        got = oracle.gemm_gelu_and_mul(x, w)
        assert int(got[0, 0]) == out, (hex(int(got[0, 0])), hex(out))


def test_projection_against_exact_rational_sums():
    rng = np.random.default_rng(7)
    x = oracle.rn16_array(rng.normal(0, 1, (3, 40)))
    w = oracle.rn16_array(rng.normal(0, 0.2, (5, 40)))
    exact, _, _ = oracle.gate_up_bf16(x, w)
    for t in range(3):
        for n in range(5):
            s = sum(Fraction(_val(a)) * Fraction(_val(b)) for a, b in zip(x[t], w[n]))
            r = round_fraction(s, 8, -126, 127)
            assert _val(int(exact[t, n])) == float(r), (t, n)


def test_identity_weights_reduce_to_plain_geglu():
    C = 64
    x = bits(W.normal_bf16((50, C), 31, 0, std=2.0))
    eye = np.zeros((C, C), np.uint16)
    eye[np.arange(C), np.arange(C)] = 0x3F80
    w = np.concatenate([eye, eye], axis=0)                # gate = up = x
    np.testing.assert_array_equal(oracle.gemm_gelu_and_mul(x, w), oracle.gelu_and_mul(x, x))
    zero = np.zeros_like(w)
    assert not oracle.gemm_gelu_and_mul(x, zero).any()     # up * gelu(0) = +0


def test_bounds_hold_for_fp32_sums_in_any_order():
    rng = np.random.default_rng(11)
    T, C, N = 6, 512, 8
    x = bits(W.normal_bf16((T, C), 12, 0))
    w = bits(W.normal_bf16((N, C), 12, 1, std=C ** -0.5))
    eps = C * 2.0 ** -23
    exact, lo, hi = oracle.gate_up_bf16(x, w, eps)
    xf = oracle.bits_to_f64(x).astype(np.float32)
    wf = oracle.bits_to_f64(w).astype(np.float32)
    key = lambda u: np.where(u & 0x8000, 0x8000 - (u.astype(np.int64) & 0x7FFF),
                             0x8000 + u.astype(np.int64))
    for _ in range(20):
        perm = rng.permutation(C)
        prods = (xf[:, None, perm] * wf[None, :, perm]).astype(np.float32)  # exact products
        acc = np.zeros((T, N), np.float32)
        for c in range(C):                                   # sequential fp32 sum
            acc = (acc + prods[:, :, c]).astype(np.float32)
        got = bits(torch.from_numpy(acc).to(torch.bfloat16))
        assert (key(lo) <= key(got)).all() and (key(got) <= key(hi)).all()
    assert (key(lo) <= key(exact)).all() and (key(exact) <= key(hi)).all()
