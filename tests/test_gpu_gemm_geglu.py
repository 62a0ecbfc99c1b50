"""GEGLU in the epilogue of the gate_up projection (tcgen05 GEMM) against the oracle.

The projection is accumulated in fp32 by the tensor cores in an unspecified
order, so two kinds of case:
  - inputs whose partial sums are all exact in fp32 (small multiples of 2^-6):
    every order gives the exact sum, and the result must equal the oracle bit
    for bit;
  - realistic values (x ~ N(0, 1), w ~ U(-1/sqrt C, 1/sqrt C), the nn.Linear
    default): the kernel also stores the rounded projection (gate_up); every
    gate and up value must lie within the bf16 rounding of an fp32
    accumulation with error below (C + 1) * 2^-23 * sum|x w| (the oracle's
    bounds), at most 1% of them may differ from the rounding of the exact sum,
    and the output must be the GEGLU of the stored gate and up, bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import diffusion_transformer_elementwise_rotate_b300 as dt
from diffusion_transformer_elementwise_rotate_b300 import _capi
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _compare import assert_bitexact

pytestmark = pytest.mark.gpu
bits = oracle.bf16_bits


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dt.load()
    torch.cuda.init()


def _grid_values(shape, seed):
    """bf16 values k * 2^-6, k in [-8, 8]: products are multiples of 2^-12 and
    sums of up to 2^13 of them stay exact in fp32."""
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(-8, 9, shape, generator=g).to(torch.float32)
    return (k * 2.0 ** -6).to(torch.bfloat16)


def _run(x, w, out=None):
    got = dt.gemm_gelu_and_mul(x.cuda(), w.cuda(), out=out)
    torch.cuda.synchronize()
    return got


def _check_workspace_error_word():
    ws = dt.api._ws_cache[("gemm_geglu", torch.cuda.current_device(),
                           torch.cuda.current_stream().cuda_stream)]
    err = int(ws[17152:17156].view(torch.int32).item())
    assert err == 0, f"a wait inside the kernel ran out of time (code {err})"


# T <= 128 runs one CTA per 128-row tile; larger T runs CTA pairs (256-row
# tiles): T = 129 leaves the second CTA of the pair one valid row, and F = 40 or
# 264 ends the output inside a 32-column store block.
@pytest.mark.parametrize("T,C,F", [(128, 64, 128), (300, 512, 256), (257, 1000, 200),
                                   (33, 4096, 384), (1, 8, 8), (129, 192, 40),
                                   (255, 320, 264), (640, 128, 1000)])
def test_exact_inputs_bitexact(T, C, F):
    x = _grid_values((T, C), T + C)
    w = _grid_values((2 * F, C), F + 7)
    gu = torch.empty((T, 2 * F), dtype=torch.bfloat16, device="cuda")
    got = dt.gemm_gelu_and_mul(x.cuda(), w.cuda(), gate_up=gu)
    torch.cuda.synchronize()
    assert_bitexact(bits(got), oracle.gemm_gelu_and_mul(bits(x), bits(w)), f"T={T} C={C} F={F}")
    assert_bitexact(bits(gu), oracle.gate_up_bf16(bits(x), bits(w))[0], "gate_up")
    _check_workspace_error_word()


def test_every_gate_value_through_the_epilogue():
    # x[t] = e_0, so gate[t, f] = w[f, 0]: the gate rows carry every bf16 bit
    # pattern once, the up rows are 1.  The projection sums 1 * w[f, 0] with
    # 0 * 0 terms, so -0 weights give +0 (IEEE), as in the oracle.
    T, C, F = 3, 64, 1 << 16
    x = torch.zeros((T, C), dtype=torch.bfloat16)
    x[:, 0] = 1.0
    w = torch.zeros((2 * F, C), dtype=torch.bfloat16)
    w[:F, 0] = torch.from_numpy(np.arange(F, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    w[F:, 0] = 1.0
    got = _run(x, w)
    assert_bitexact(bits(got), oracle.gemm_gelu_and_mul(bits(x), bits(w)), "every gate value")


def _realistic(T, C, F, seed):
    x = W.normal_bf16((T, C), seed, 0)
    g = torch.Generator().manual_seed(seed * 7 + 1)
    bound = 1.0 / math.sqrt(C)
    w = (torch.rand((2 * F, C), generator=g) * 2 * bound - bound).to(torch.bfloat16)
    return x, w


def _key(u):
    u = u.astype(np.int64)
    k = np.where(u & 0x8000, 0x8000 - (u & 0x7FFF), 0x8000 + u)
    return np.where((u & 0x7FFF) == 0, 0x8000, k)


def _check_projection(out, gu, xb, wb, what, max_diff_fraction=1e-2):
    """out, gu: the kernel's outputs (uint16); xb, wb: its inputs (rows of x,
    rows of w as gate rows then up rows)."""
    C = xb.shape[1]
    F = wb.shape[0] // 2
    eps = (C + 1) * 2.0 ** -23
    exact, lo, hi = oracle.gate_up_bf16(xb, wb, eps)
    k = _key(gu)
    assert ((_key(lo) <= k) & (k <= _key(hi))).all(), f"{what}: gate_up outside the fp32 bounds"
    n = int((gu != exact).sum())
    assert n <= max_diff_fraction * gu.size, f"{what}: {n} of {gu.size} projections differ"
    assert_bitexact(out, oracle.gelu_and_mul(gu[:, :F], gu[:, F:]), f"{what}: epilogue")
    print(f"{what}: {n} of {gu.size} gate/up values differ from the exactly rounded projection")
    return n


@pytest.mark.parametrize("T,C,F", [(256, 2048, 512), (200, 5120, 256)])
def test_realistic_inputs_within_accumulation_bounds(T, C, F):
    x, w = _realistic(T, C, F, T + F)
    gu = torch.empty((T, 2 * F), dtype=torch.bfloat16, device="cuda")
    out = dt.gemm_gelu_and_mul(x.cuda(), w.cuda(), gate_up=gu)
    torch.cuda.synchronize()
    _check_projection(bits(out), bits(gu), bits(x), bits(w), f"T={T} C={C} F={F}")
    _check_workspace_error_word()


def test_video_layer_mlp_sampled_outputs():
    # the video layer's MLP: x (32760, 5120), w (2 x 13824, 5120)
    T, C, F = 32760, 5120, 13824
    x, w = _realistic(T, C, F, 3)
    gu = torch.empty((T, 2 * F), dtype=torch.bfloat16, device="cuda")
    out = dt.gemm_gelu_and_mul(x.cuda(), w.cuda(), gate_up=gu)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    cols = np.unique(np.concatenate([[0, F - 1], rng.choice(F, 94, replace=False)]))
    wb = bits(w)
    wsub = np.concatenate([wb[cols], wb[F + cols]], axis=0)
    gsel = np.concatenate([cols, F + cols])
    r = torch.from_numpy(rows).cuda()
    _check_projection(bits(out[r])[:, cols], bits(gu[r])[:, gsel], bits(x)[rows], wsub,
                      "video MLP sample")
    _check_workspace_error_word()


def test_strided_output_and_caller_workspace():
    T, C, F = 130, 256, 136
    x = _grid_values((T, C), 1)
    w = _grid_values((2 * F, C), 2)
    big = torch.full((T, F + 24), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:, 8:8 + F]
    n = int(_capi.load().dtrot_gemm_gelu_and_mul_workspace_bytes())
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")  # garbage, incl. the error word
    dt.gemm_gelu_and_mul(x.cuda(), w.cuda(), out=out, workspace=ws)
    torch.cuda.synchronize()
    assert_bitexact(bits(out), oracle.gemm_gelu_and_mul(bits(x), bits(w)), "strided out")
    assert (big[:, :8] == 7.0).all() and (big[:, 8 + F:] == 7.0).all()
    assert int(ws[17152:17156].view(torch.int32).item()) == 0


# A stalled pipeline: the diagnostic entry point withholds the loads of each
# CTA's last stage, so the MMA thread's bounded wait for that stage runs out
# (about a second; nothing ever loads it).  The kernel must come back on its
# own with bit 2 (a loaded-stage wait ran out) in its error word, the API must
# raise when asked to check, and the next call on the same workspace must be
# clean and exact: the device stays usable.  T = 100 runs single CTAs, T = 512
# CTA pairs.
@pytest.mark.parametrize("T,C,F", [(100, 256, 128), (512, 256, 256)])
def test_stalled_pipeline_is_reported_and_the_device_stays_usable(T, C, F):
    import time
    x = _grid_values((T, C), 11).cuda()
    w = _grid_values((2 * F, C), 12).cuda()
    n = int(_capi.load().dtrot_gemm_gelu_and_mul_workspace_bytes())
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.empty((T, F), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    dt.gemm_gelu_and_mul(x, w, out=out, workspace=ws, _withhold_last_stage=True)
    word = dt.api.gemm_error_word(ws)
    elapsed = time.time() - t0
    assert word & 2, f"error word {word:#x}: the withheld stage's wait did not report"
    assert word & ~0x7 == 0, f"error word {word:#x}"
    assert elapsed < 30.0
    with pytest.raises(_capi.DtrotKernelError):
        dt.gemm_gelu_and_mul(x, w, out=out, workspace=ws, check=True, _withhold_last_stage=True)
    got = dt.gemm_gelu_and_mul(x, w, out=out, workspace=ws, check=True)
    assert dt.api.gemm_error_word(ws) == 0
    assert_bitexact(bits(got), oracle.gemm_gelu_and_mul(bits(x.cpu()), bits(w.cpu())),
                    "the call after the stall")
