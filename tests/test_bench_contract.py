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
