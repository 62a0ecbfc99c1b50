"""The layer step captured in a CUDA graph gives the same bits as eager calls.

The benchmark times the step (cos/sin tables, RoPE on q and k, GEGLU, two
RMSNorm+residual calls) as a replayed CUDA graph, in which the kernels keep
their programmatic-dependent launch edges.  Here the tiny and image layers'
steps are captured, replayed twice (the residuals carry over from one replay
to the next, as in consecutive layers), and every output is compared bit for
bit with the same sequence of eager calls, and the first replay with the
oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import diffusion_transformer_elementwise_rotate_b300 as dt
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _compare import assert_bitexact, assert_within_tolerance

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))
bits = oracle.bf16_bits


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dt.load()
    torch.cuda.init()


def _tensors(wl):
    h = {"freqs": W.freqs_for(wl), "q": W.rope_inputs(wl, "q"), "k": W.rope_inputs(wl, "k"),
         "gu": W.geglu_inputs(wl)}
    h["x1"], h["r1"], h["w"] = W.rmsnorm_inputs(wl, False)
    h["x2"], h["r2"], _ = W.rmsnorm_inputs(wl, True)
    return h


def _device_set(h, wl):
    d = {k: v.cuda() for k, v in h.items()}
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    d.update({"cos": e((wl.B * wl.S, wl.rot)), "sin": e((wl.B * wl.S, wl.rot)),
              "qo": e(tuple(h["q"].shape)), "ko": e(tuple(h["k"].shape)),
              "ff": e((wl.T_ff, wl.F)), "y1": e((wl.T_norm, wl.C)), "y2": e((wl.T_norm, wl.C))})
    return d


def _step(d, F):
    dt.rope_cos_sin_precompute(d["freqs"], d["cos"], d["sin"])
    dt.rope_rotate_half(d["q"], d["cos"], d["sin"], out=d["qo"])
    dt.rope_rotate_half(d["k"], d["cos"], d["sin"], out=d["ko"])
    dt.gelu_and_mul(d["gu"][:, :F], d["gu"][:, F:], out=d["ff"])
    dt.rmsnorm_residual(d["x1"], d["r1"], d["w"], EPS, out=d["y1"])
    dt.rmsnorm_residual(d["x2"], d["r2"], d["w"], EPS, out=d["y2"])


OUTS = ("cos", "sin", "qo", "ko", "ff", "y1", "y2", "r1", "r2")


@pytest.mark.parametrize("name", ["tiny", "image"])
def test_graph_replay_matches_eager_calls_and_the_oracle(name):
    wl = W.WORKLOADS[name]
    h = _tensors(wl)
    eager, graphed = _device_set(h, wl), _device_set(h, wl)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    scratch = _device_set(h, wl)
    with torch.cuda.stream(side):
        _step(scratch, wl.F)   # first calls (workspace, attributes) outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(graphed, wl.F)
    torch.cuda.synchronize()
    for rep in range(2):
        g.replay()
        _step(eager, wl.F)
        torch.cuda.synchronize()
        for k in OUTS:
            assert_bitexact(bits(graphed[k]), bits(eager[k]), f"{name} replay {rep} {k}")
        if rep == 0:
            ec, es = oracle.rope_cos_sin(h["freqs"].numpy())
            assert_bitexact(bits(graphed["cos"]), ec, "cos")
            assert_bitexact(bits(graphed["qo"]), oracle.rope_rotate_half(bits(h["q"]), ec, es),
                            "rope q")
            assert_bitexact(bits(graphed["ko"]), oracle.rope_rotate_half(bits(h["k"]), ec, es),
                            "rope k")
            assert_bitexact(bits(graphed["ff"]), oracle.gelu_and_mul_fused(bits(h["gu"])), "geglu")
            he, ye = oracle.rmsnorm_residual(bits(h["x1"]), bits(h["r1"]), bits(h["w"]), EPS)
            assert_bitexact(bits(graphed["r1"]), he, "residual")
            assert_within_tolerance(bits(graphed["y1"]), ye, "rmsnorm")
