"""The benchmark's reference arm (the oracle on host cores) keeps the JSON line
contract, on CPU: one line with the arm's metric, unit, config and the
cpu_baseline / e2e objects, and ranks other than 0 exit without work."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *args):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    p = _run({}, "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3")
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    from diffusion_transformer_elementwise_rotate_b300 import workloads as W
    wl = W.WORKLOADS["tiny"]
    assert d["config"] == bench.config_for(wl, sum(bench.step_bytes(wl, W).values()),
                                           "host cores")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == "GB/s" and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    p = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"},
             "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3")
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


def test_source_hash_ignores_comments_and_whitespace():
    import bench
    a = 'int f(int x) { // doubles\n  return 2 * x; /* fast */ }\nconst char* s = "// kept";\n'
    b = 'int f(int x) {\n    return 2 * x;   }\n   const char* s = "// kept";'
    c = 'int f(int x) { return 3 * x; } const char* s = "// kept";'
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
    assert '"// kept"' in bench.code_text(a)


def test_sample_parity_checks_the_sampled_rows():
    """The benchmark's check of the GPU outputs against the oracle on its CPU
    sample, run here on outputs the oracle made for the whole layer: they
    agree; one bit flipped inside the sample is counted, one outside it is not.
    B = 2 puts the second sequence's table rows at S + s in the layer and at
    tok + s in the sample."""
    import dataclasses

    import torch

    import oracle
    from diffusion_transformer_elementwise_rotate_b300 import workloads as W
    wl = dataclasses.replace(W.WORKLOADS["tiny"], name="tiny_b2", B=2, S=64, grid=(64,),
                             T_ff=48, T_norm=40)
    layer = bench.Layer(wl, W, torch.device("cpu"))
    full = bench.oracle_step(
        oracle, bench.oracle_sample_inputs(oracle, layer.h_in, wl.S, wl.T_ff, wl.T_norm), wl.F)
    assert set(full) == set(layer.out_names)
    for n, a in full.items():
        layer.h_out[n].copy_(oracle.from_bits(a).reshape(layer.h_out[n].shape))
    tok, rf, rn = 16, 20, 10
    ref = bench.oracle_step(oracle, bench.oracle_sample_inputs(oracle, layer.h_in, tok, rf, rn),
                            wl.F)
    res = bench.sample_parity(ref, layer, wl, tok, rf, rn)
    assert res["bit_exact"]
    assert res["outputs"]["cos"]["elements"] == wl.B * tok * wl.rot
    assert res["outputs"]["q_out"]["elements"] == wl.B * tok * wl.H * wl.D
    assert res["outputs"]["ff_out"]["elements"] == rf * wl.F
    assert res["outputs"]["y2"]["elements"] == rn * wl.C
    layer.h_out["cos"].view(torch.int16)[wl.S + 3, 5] ^= 1      # b = 1, s = 3: sampled
    layer.h_out["ff_out"].view(torch.int16)[rf + 1, 0] ^= 1     # beyond the sampled rows
    layer.h_out["k_out"].view(torch.int16)[1, tok, 0, 0] ^= 1   # position tok: not sampled
    res = bench.sample_parity(ref, layer, wl, tok, rf, rn)
    assert not res["bit_exact"]
    diff = {n: o["differing"] for n, o in res["outputs"].items()}
    assert diff == {n: int(n == "cos") for n in layer.out_names}
    assert res["outputs"]["cos"]["max_ulp"] == 1


def test_step_accounting_of_both_rope_forms():
    """The step's calls and bytes: one q+k launch reads the tables once where two
    rope_rotate_half calls read them twice; the GEGLU activation table is its own
    launch; a sample of the whole layer counts the whole step."""
    from diffusion_transformer_elementwise_rotate_b300 import workloads as W
    wl = W.WORKLOADS["video"]
    qk, sep = bench.step_ops("qk"), bench.step_ops("separate")
    assert qk[:2] == list(bench.PER_FORWARD) and qk[-1] == bench.DOMINANT
    assert qk == ["rope_cos_sin_precompute", "gelu_table_build", "rmsnorm_residual_attn",
                  "rope_rotate_half_qk", "rmsnorm_residual_ffn", "gelu_and_mul"]
    assert sep[3:5] == ["rope_rotate_half_q", "rope_rotate_half_k"] and len(sep) == len(qk) + 1
    assert bench.launches_per_step("qk") == 6 and bench.launches_per_step("separate") == 7
    bq, bs = bench.step_bytes(wl, W, "qk"), bench.step_bytes(wl, W, "separate")
    assert list(bq) == qk and list(bs) == sep
    tok = wl.B * wl.S
    assert sum(bs.values()) - sum(bq.values()) == 4 * tok * wl.rot  # one more table read
    assert bq["rope_rotate_half_qk"] == 2 * 4 * tok * wl.H * wl.D + 4 * tok * wl.rot
    assert bq["gelu_table_build"] == 2 * 65536
    whole = bench.sampled_bytes(bq, wl, wl.S, wl.T_ff, wl.T_norm)
    assert whole == sum(bq.values())
    half = bench.sampled_bytes(bq, wl, wl.S // 2, wl.T_ff // 2, wl.T_norm // 2)
    assert abs(half - (sum(bq.values()) - bq["gelu_table_build"]) / 2
               - bq["gelu_table_build"]) < 1e-3 * sum(bq.values())
