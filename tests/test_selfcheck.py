"""The opt-in first-call self-check (selfcheck.py).

CPU: its comparison rule, with differences planted in the data it is given,
and its plain-torch references pinned to the oracle on CPU tensors.
GPU: every op runs with the check enabled, each (op, shape) key is checked
once, and the kernels pass it.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_elementwise_rotate_b300 import selfcheck as sc
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _compare import assert_bitexact, assert_within_tolerance

bits = oracle.bf16_bits


def _bf(a):
    return oracle.from_bits(np.asarray(a, dtype=np.uint16))


def test_compare_accepts_equal_and_tolerated_differences():
    x = W.normal_bf16((1000, 100), 1, 0)
    assert sc.compare("same", x, x.clone(), exact=True) == 0
    y = bits(x).copy()
    y[3, 4] += 1                      # one element one bf16 step away (magnitude grows)
    assert sc.compare("one step", _bf(y), x, exact=False) == 1
    z = np.zeros(4, np.uint16)
    z[1] = 0x8000                     # -0 against +0
    z[2] = z[3] = 0x7FC1              # NaN against NaN (other payload)
    ref = np.array([0, 0, 0x7FC0, 0xFFC0], np.uint16)
    assert sc.compare("zeros and NaNs", _bf(z), _bf(ref), exact=True) == 0


def test_compare_rejects_planted_differences():
    x = W.normal_bf16((1000, 100), 2, 0)
    y = bits(x).copy()
    y[0, 0] += 1
    with pytest.raises(sc.SelfCheckError):
        sc.compare("exact", _bf(y), x, exact=True)
    y[0, 0] += 1                      # now two steps away
    with pytest.raises(sc.SelfCheckError):
        sc.compare("two steps", _bf(y), x, exact=False)
    y = bits(x).copy()
    y.flat[:11] += 1                  # 11 of 100000 > 0.01%
    with pytest.raises(sc.SelfCheckError):
        sc.compare("too many", _bf(y), x, exact=False)
    y = bits(x).copy()
    y[5, 5] = 0x7FC0                  # NaN where the reference has a number
    with pytest.raises(sc.SelfCheckError):
        sc.compare("nan", _bf(y), x, exact=False)
    with pytest.raises(sc.SelfCheckError):
        sc.compare("shape", x[:10], x[:11], exact=False)


def test_want_checks_each_key_once():
    sc.enable()
    sc.reset()
    try:
        t = torch.zeros(4, 8)
        assert sc.want("op", t) is not None
        assert sc.want("op", t) is None
        assert sc.want("op", torch.zeros(4, 9)) is not None
        assert len(sc.checked()) == 2
    finally:
        sc.disable()
        sc.reset()
    assert sc.want("op", torch.zeros(1)) is None


def test_references_match_the_oracle_on_cpu():
    wl = W.WORKLOADS["tiny"]
    freqs = W.freqs_for(wl)
    ec, es = oracle.rope_cos_sin(freqs.numpy())
    rc, rs = sc.ref_tables(freqs)
    assert_within_tolerance(bits(rc), ec, "ref cos")
    assert_within_tolerance(bits(rs), es, "ref sin")
    x = W.rope_inputs(wl, "q")
    got = sc.ref_rope(x, _bf(ec), _bf(es))
    assert_bitexact(bits(got), oracle.rope_rotate_half(bits(x), ec, es), "ref rope")
    gate = np.arange(1 << 16, dtype=np.uint16).reshape(256, 256)
    up = bits(W.normal_bf16((256, 256), 3, 3))
    assert_within_tolerance(bits(sc.ref_geglu(_bf(gate), _bf(up))),
                            oracle.gelu_and_mul(gate, up), "ref geglu")
    xn, r, w = W.rmsnorm_inputs(wl)
    h, y = sc.ref_rmsnorm(xn, r, w, 1e-6)
    h_exp, y_exp = oracle.rmsnorm_residual(bits(xn), bits(r), bits(w), float(np.float32(1e-6)))
    assert_bitexact(bits(h), h_exp, "ref residual")
    assert_within_tolerance(bits(y), y_exp, "ref rmsnorm")


@pytest.mark.gpu
def test_every_op_passes_the_check_on_the_gpu():
    import diffusion_transformer_elementwise_rotate_b300 as dt
    dt.load()
    sc.enable()
    sc.reset()
    try:
        for name in ("tiny", "image"):
            wl = W.WORKLOADS[name]
            freqs = W.freqs_for(wl).cuda()
            c, s = dt.rope_cos_sin_precompute(freqs)
            q, k = W.rope_inputs(wl, "q").cuda(), W.rope_inputs(wl, "k").cuda()
            dt.rope_rotate_half(q, c, s)
            dt.rope_rotate_half(q, c, s, out=q)                 # in place
            dt.rope_rotate_half_qk_(q, k, cos=c, sin=s)
            dt.rope_rotate_half_qk_(q, k, freqs=freqs)
            dt.rope_rotate_half_qk(q, k, cos=c, sin=s)          # out of place
            dt.rope_rotate_half_qk(q, k, freqs=freqs)
            dt.gelu_and_mul_fused(W.geglu_inputs(wl).cuda())
            x, r, w = (t.cuda() for t in W.rmsnorm_inputs(wl))
            dt.rmsnorm_residual(x, r, w, 1e-6)
            n = len(sc.checked())
            dt.rmsnorm_residual(x, r, w, 1e-6)                 # same key: not checked again
            assert len(sc.checked()) == n
            xm = W.normal_bf16((300, 512), 41, 0).cuda()
            wm = (torch.rand((2 * 256, 512), device="cuda") * 2 - 1).mul(512 ** -0.5)
            dt.gemm_gelu_and_mul(xm, wm.to(torch.bfloat16))
        ops = {k[0] for k in sc.checked()}
        assert ops == {"rope_cos_sin_precompute", "rope_rotate_half", "rope_rotate_half_qk",
                       "rope_rotate_half_qk_out", "gelu_and_mul", "rmsnorm_residual",
                       "gemm_gelu_and_mul"}
    finally:
        sc.disable()
        sc.reset()
