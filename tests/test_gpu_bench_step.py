"""The benchmark's layer step as it is timed: the per-forward tables (cos/sin
and the GEGLU activation table) on a side branch of a CUDA graph, beside the
pre-attention norm, then RoPE, the pre-FFN norm and GEGLU.  Replayed twice
(the residuals carry over, as in consecutive layers), it writes the same bits
as the same calls made one after another on one stream, and its first replay
matches the oracle on the whole layer, through the benchmark's own
element-by-element check."""
import pytest
import torch

import bench
import oracle
import diffusion_transformer_elementwise_rotate_b300 as dt
from diffusion_transformer_elementwise_rotate_b300 import workloads as W

pytestmark = pytest.mark.gpu
INEXACT = ("ff_out", "y1", "y2")  # GEGLU and RMSNorm: within 1 ulp on at most 0.01%


@pytest.mark.parametrize("rope", ["qk", "separate"])
@pytest.mark.parametrize("name", ["tiny", "image"])
def test_timed_step_matches_serial_calls_and_the_oracle(name, rope):
    dt.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = W.WORKLOADS[name]
    timed = bench.Layer(wl, W, dev, rope=rope)
    serial = bench.Layer(wl, W, dev, rope=rope, serial=True)
    g = bench.step_graph(dt, timed, 1)
    for layer in (timed, serial):
        for r in ("r1", "r2"):
            layer.d[r].copy_(layer.h_in[r])
    torch.cuda.synchronize()
    for rep in range(2):
        g.replay()
        serial.step(dt)
        torch.cuda.synchronize()
        for n in timed.out_names:
            assert torch.equal(timed.d[n].view(torch.int16), serial.d[n].view(torch.int16)), \
                f"{name} {rope} replay {rep}: {n}"
        if rep == 0:
            timed.d2h()
            torch.cuda.synchronize()
            inp = bench.oracle_sample_inputs(oracle, timed.h_in, wl.S, wl.T_ff, wl.T_norm)
            ref = bench.oracle_step(oracle, inp, wl.F)
            res = bench.sample_parity(ref, timed, wl, wl.S, wl.T_ff, wl.T_norm)
            for n, o in res["outputs"].items():
                if n in INEXACT:
                    assert o["max_ulp"] <= 1 and o["differing"] <= 1e-4 * o["elements"], (n, o)
                else:
                    assert o["differing"] == 0, (n, o)
