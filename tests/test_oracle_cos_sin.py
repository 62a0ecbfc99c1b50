"""Pins for the oracle's rotary cos/sin tables.

Reading pinned: each entry is RN16(RN32(cos f)) (fp32 cos, then bf16), at row
b*S + s of the (B*S, rot_dim) output, as the ERNIE-Image fusion page's section 1
describes (permute (S,B,1,R) -> (B,S,1,R), cos/sin, cast, reshape).  The values
are checked against mpmath at 50 digits followed by exact rational rounding.
"""
import mpmath
import numpy as np
import torch

import oracle
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _exact import rn16_of_rn32_bits

mpmath.mp.dps = 50


def _exact_bits(f32_vals):
    cs, ss = [], []
    for v in f32_vals:
        a = mpmath.mpf(float(v))
        cs.append(rn16_of_rn32_bits(mpmath.cos(a)))
        ss.append(rn16_of_rn32_bits(mpmath.sin(a)))
    return np.array(cs, dtype=np.uint16), np.array(ss, dtype=np.uint16)


def test_zero_angle():
    cos, sin = oracle.rope_cos_sin(np.zeros((1, 1, 1, 2), np.float32))
    assert cos.tolist() == [[0x3F80, 0x3F80]] and sin.tolist() == [[0, 0]]


def test_tiny_table_against_mpmath():
    wl = W.WORKLOADS["tiny"]
    freqs = W.freqs_for(wl).numpy()
    cos, sin = oracle.rope_cos_sin(freqs)
    flat = freqs.reshape(-1)  # B = 1: row s == freqs[s, 0, 0, :]
    uniq, inv = np.unique(flat, return_inverse=True)
    ec, es = _exact_bits(uniq)
    assert np.array_equal(cos.reshape(-1), ec[inv])
    assert np.array_equal(sin.reshape(-1), es[inv])


def test_random_angles_against_mpmath():
    rng = np.random.default_rng(7)
    a = np.concatenate([rng.uniform(-60, 60, 6000), rng.uniform(-1e4, 1e4, 3000),
                        rng.uniform(-1e-3, 1e-3, 1000)]).astype(np.float32)
    cos, sin = oracle.rope_cos_sin(a.reshape(-1, 1, 1, 1))
    ec, es = _exact_bits(a)
    assert np.array_equal(cos.reshape(-1), ec)
    assert np.array_equal(sin.reshape(-1), es)


def test_row_layout_is_b_major():
    S, B, R = 5, 3, 4
    freqs = (np.arange(S * B * R, dtype=np.float32) * 0.01).reshape(S, B, 1, R)
    cos, sin = oracle.rope_cos_sin(freqs)
    ref = torch.from_numpy(freqs).permute(1, 0, 2, 3).reshape(-1, R).numpy()
    ec, es = _exact_bits(ref.reshape(-1))
    assert np.array_equal(cos.reshape(-1), ec)
    assert np.array_equal(sin.reshape(-1), es)


def test_against_torch_cpu_cast_is_close():
    # torch.cos in fp32 is not correctly rounded, so a few entries may differ;
    # this is the reported gap between the eager chain and exact math.
    wl = W.WORKLOADS["image"]
    freqs = W.freqs_for(wl)
    cos, sin = oracle.rope_cos_sin(freqs.numpy())
    tc = oracle.bf16_bits(torch.cos(freqs.permute(1, 0, 2, 3)).to(torch.bfloat16)).reshape(cos.shape)
    ts = oracle.bf16_bits(torch.sin(freqs.permute(1, 0, 2, 3)).to(torch.bfloat16)).reshape(sin.shape)
    diff = np.count_nonzero(tc != cos) + np.count_nonzero(ts != sin)
    assert diff <= 1e-4 * 2 * cos.size
    # where they differ, it is by one bf16 step
    for a, b in ((tc, cos), (ts, sin)):
        d = np.abs(a.astype(np.int32) - b.astype(np.int32))
        assert d.max() <= 1
