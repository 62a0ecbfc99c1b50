"""The C ABI from plain C: tests/c_caller/dtrot_c_caller.c includes dtrot.h,
takes its device memory from the CUDA runtime and calls the library without
Python or torch on its path.

On CPU: the header and the caller compile as C11 with all warnings as errors
and link against libdtrot.so.  On the GPU: the caller runs the tables, RoPE,
GEGLU (with a workspace and without one) and RMSNorm on seeded inputs written
by this test, and its outputs match the oracle.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_elementwise_rotate_b300 import build as dbuild
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _compare import assert_bitexact, assert_within_tolerance

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller", "dtrot_c_caller.c")
PKG = os.path.join(ROOT, "diffusion_transformer_elementwise_rotate_b300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    dbuild.build()
    exe = os.path.join(out_dir, "dtrot_c_caller")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-o", exe, SRC, "-L", PKG, "-ldtrot", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{PKG}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_header_and_c_caller_compile_as_c(tmp_path):
    assert os.path.exists(_compile(str(tmp_path)))


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.gpu
def test_plain_c_caller_matches_the_oracle(tmp_path):
    exe = _compile(str(tmp_path))
    B, S, H, D, R = 2, 37, 3, 64, 48
    T, F, C = 21, 200, 264
    freqs = W.freqs_1d(S, B, R).numpy()
    x = _bits(W.normal_bf16((B, S, H, D), 500, 0))
    gu = _bits(W.normal_bf16((T, 2 * F), 500, 2))
    hx = _bits(W.normal_bf16((T, C), 500, 4))
    hr = _bits(W.normal_bf16((T, C), 500, 5, std=2.0))
    hw = _bits(W.normal_bf16((C,), 500, 6, mean=1.0, std=0.316))
    d = str(tmp_path)
    for name, a in (("freqs.f32", freqs), ("x.bf16", x), ("gate_up.bf16", gu), ("hx.bf16", hx),
                    ("hr.bf16", hr), ("hw.bf16", hw)):
        a.tofile(os.path.join(d, name))
    r = subprocess.run([exe, d, *map(str, (B, S, H, D, R, T, F, C))], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    load = lambda n, shape: np.fromfile(os.path.join(d, n), dtype=np.uint16).reshape(shape)  # noqa: E731
    ec, es = oracle.rope_cos_sin(freqs)
    assert_bitexact(load("cos.bf16", ec.shape), ec, "cos")
    assert_bitexact(load("sin.bf16", es.shape), es, "sin")
    assert_bitexact(load("rope.bf16", x.shape), oracle.rope_rotate_half(x, ec, es), "rope")
    for n in ("rope_qk_q.bf16", "rope_qk_k.bf16"):  # one out-of-place q+k launch, tail copied
        assert_bitexact(load(n, x.shape), oracle.rope_rotate_half(x, ec, es), n)
    ref = oracle.gelu_and_mul(gu[:, :F], gu[:, F:])
    assert_within_tolerance(load("geglu.bf16", (T, F)), ref, "geglu")
    assert_bitexact(load("geglu_noalloc.bf16", (T, F)), load("geglu.bf16", (T, F)),
                    "noalloc equals the workspace call")
    h, y = oracle.rmsnorm_residual(hx, hr, hw, float(np.float32(1e-6)))
    assert_bitexact(load("residual.bf16", (T, C)), h, "residual")
    assert_within_tolerance(load("norm.bf16", (T, C)), y, "rmsnorm")
