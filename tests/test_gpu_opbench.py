"""opbench (one op alone, the case behind the per-kernel DRAM captures) runs
every op on the tiny layer, in CUDA graphs and eagerly, and reports
consistent figures."""
import pytest

from diffusion_transformer_elementwise_rotate_b300 import opbench

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("op", opbench.OPS)
@pytest.mark.parametrize("graph", [True, False])
def test_every_op_runs_and_reports(op, graph):
    r = opbench.run(op, "tiny", rows=None, reps=3, warmup=1, graph=graph)
    assert r["op"] == op and r["reps"] == 3 and r["graph"] == graph
    assert 0 < r["launch_ms_min"] <= r["launch_ms_median"] <= r["launch_ms_max"]
    assert r["back_to_back_ms"] > 0 and r["rate"] > 0 and r["rate_back_to_back"] > 0
    assert r["work"] > 0 and r["work_unit"] in ("B", "flop")


def test_rmsnorm_width_option():
    # a width no workload has (the one-warp-per-row kernel), rows given exactly
    r = opbench.run("rmsnorm", "tiny", rows=300, reps=3, warmup=1, graph=True, cols=1152)
    assert r["case"] == "rmsnorm_residual (300, 1152)"
    assert r["work"] == 8 * 300 * 1152 + 2 * 1152 and r["rate"] > 0
