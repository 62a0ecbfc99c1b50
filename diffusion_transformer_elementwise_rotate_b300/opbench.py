"""Time one op of the hot path on its own, with only that op's tensors on the
device: the standalone case behind the per-kernel DRAM-traffic captures and
the per-launch timing spread.

    python -m diffusion_transformer_elementwise_rotate_b300.opbench --op OP
        [--workload video] [--rows N] [--cols C] [--reps K] [--warmup W]

OP is one of
  tables      rope_cos_sin_precompute on the workload's (S, B, 1, rot) angles
  rope        rope_rotate_half on q (B, S, H, D), out of place
  rope_qk     rope_rotate_half_qk_ on q and k in place, from the tables
  rope_qk_out rope_rotate_half_qk on q and k into separate outputs, from the tables
  rope_qk_angles   the same, cos/sin evaluated in the kernel from the angles
  geglu       gelu_and_mul on a (T, 2F) gate_up buffer (activation table + stream)
  geglu_table gelu_and_mul with a prebuilt activation table (the stream alone)
  rmsnorm     rmsnorm_residual on (T, C)
  gemm        gemm_gelu_and_mul: x (T, C) times w (2F, C)^T with GEGLU in the epilogue

--rows caps the op's row count (tokens for the RoPE ops, T for the others), so
a capture can hold a slice of a layer that still exceeds the 126 MB L2.
--cols sets the RMSNorm width C (and, with --rows, its row count exactly), for
widths no workload has (the one-warp-per-row kernel takes C <= 1280).
Inputs are drawn on the device (torch's CUDA generator, seed 0) with the
workload's distributions: timing does not depend on the values, and drawing a
few GB on the host would dominate a short run.  Every launch is bracketed by
CUDA events; the line reports the median, min and max per launch, the mean of
the same number of launches back to back, the algorithmic bytes (or flops)
and the rates.  By default the launches run as CUDA graphs (--eager: one
Python call at a time).
"""
from __future__ import annotations

import argparse
import json
import math
import statistics

import torch

from . import api as dt
from . import workloads as W

OPS = ("tables", "rope", "rope_qk", "rope_qk_out", "rope_qk_angles", "geglu", "geglu_table",
       "rmsnorm", "gemm")


def _normal(shape, dev, g, mean=0.0, std=1.0):
    t = torch.empty(shape, dtype=torch.float32, device=dev)
    t.normal_(mean, std, generator=g)
    return t.to(torch.bfloat16)


def setup(op: str, wl: W.Workload, rows: int | None, dev, cols: int | None = None):
    """(callable running one launch of the op, algorithmic bytes or flops, unit,
    description, live tensors)."""
    g = torch.Generator(device=dev).manual_seed(0)
    if op in ("tables", "rope", "rope_qk", "rope_qk_out", "rope_qk_angles"):
        S = wl.S if rows is None else min(wl.S, max(1, rows // wl.B))
        freqs = W.freqs_for(wl)[:S].contiguous().to(dev)
        B, H, D, R = wl.B, wl.H, wl.D, wl.rot
        cos, sin = dt.rope_cos_sin_precompute(freqs)
        tok = B * S
        if op == "tables":
            return (lambda: dt.rope_cos_sin_precompute(freqs, cos, sin), tok * R * 8, "B",
                    f"cos/sin tables ({tok}, {R}) from ({S}, {B}, 1, {R}) angles",
                    (freqs, cos, sin))
        q = _normal((B, S, H, D), dev, g)
        if op == "rope":
            out = torch.empty_like(q)
            return (lambda: dt.rope_rotate_half(q, cos, sin, out=out),
                    4 * tok * H * D + 4 * tok * R, "B",
                    f"rope_rotate_half x ({B}, {S}, {H}, {D}) rot {R}, out of place",
                    (freqs, cos, sin, q, out))
        k = _normal((B, S, H, D), dev, g)
        if op == "rope_qk_out":
            qo, ko = torch.empty_like(q), torch.empty_like(k)
            return (lambda: dt.rope_rotate_half_qk(q, k, cos=cos, sin=sin, q_out=qo, k_out=ko),
                    8 * tok * H * D + 4 * tok * R, "B",
                    f"rope_rotate_half_qk q, k ({B}, {S}, {H}, {D}) rot {R}, out of place, "
                    "tables", (freqs, cos, sin, q, k, qo, ko))
        moved = 4 * tok * 2 * H * R + 4 * tok * R
        if op == "rope_qk":
            return (lambda: dt.rope_rotate_half_qk_(q, k, cos=cos, sin=sin), moved, "B",
                    f"rope_rotate_half_qk q, k ({B}, {S}, {H}, {D}) rot {R}, in place, tables",
                    (freqs, cos, sin, q, k))
        return (lambda: dt.rope_rotate_half_qk_(q, k, freqs=freqs), moved, "B",
                f"rope_rotate_half_qk q, k ({B}, {S}, {H}, {D}) rot {R}, in place, angles",
                (freqs, q, k))
    if op in ("geglu", "geglu_table"):
        T = wl.T_ff if rows is None else min(wl.T_ff, rows)
        F = wl.F
        gu = _normal((T, 2 * F), dev, g)
        out = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
        if op == "geglu":
            return (lambda: dt.gelu_and_mul(gu[:, :F], gu[:, F:], out=out), 6 * T * F, "B",
                    f"gelu_and_mul ({T}, 2x{F}), activation table built in the call",
                    (gu, out))
        tab = dt.gelu_table(dev)
        return (lambda: dt.gelu_and_mul(gu[:, :F], gu[:, F:], out=out, table=tab), 6 * T * F,
                "B", f"gelu_and_mul ({T}, 2x{F}), prebuilt activation table", (gu, out, tab))
    if op == "rmsnorm":
        T = wl.T_norm if rows is None else (rows if cols else min(wl.T_norm, rows))
        C = wl.C if cols is None else cols
        x = _normal((T, C), dev, g)
        r = _normal((T, C), dev, g, std=2.0)
        w = _normal((C,), dev, g, mean=1.0, std=math.sqrt(0.1))
        y = torch.empty_like(x)
        return (lambda: dt.rmsnorm_residual(x, r, w, W.EPS, out=y), 8 * T * C + 2 * C, "B",
                f"rmsnorm_residual ({T}, {C})", (x, r, w, y))
    if op == "gemm":
        T = wl.T_norm if rows is None else min(wl.T_norm, rows)
        C, F = wl.C, wl.F
        x = _normal((T, C), dev, g)
        w = ((torch.rand((2 * F, C), generator=g, device=dev) * 2 - 1) / math.sqrt(C)).to(
            torch.bfloat16)
        out = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
        return (lambda: dt.gemm_gelu_and_mul(x, w, out=out), 2.0 * T * C * 2 * F, "flop",
                f"gemm_gelu_and_mul x ({T}, {C}) w ({2 * F}, {C})", (x, w, out))
    raise ValueError(f"unknown op {op!r}; one of {OPS}")


def _graph(fn, n, evs=None):
    """A CUDA graph of n calls of fn (evs[i]: external events around call i)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            if evs is not None:
                evs[i][0].record()
            fn()
            if evs is not None:
                evs[i][1].record()
    torch.cuda.synchronize()
    return g


def run(op: str, workload: str = "video", rows: int | None = None, reps: int = 20,
        warmup: int = 3, graph: bool = True, cols: int | None = None) -> dict:
    """Per-launch times (events around each call) and the back-to-back rate
    (reps calls between two events).  With graph=True both run as CUDA graphs,
    so that host launch overhead never shows in the times (a short kernel
    launched from Python one call at a time can leave the GPU waiting)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    fn, work, unit, desc, _live = setup(op, W.WORKLOADS[workload], rows, dev, cols)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True, external=graph),
            torch.cuda.Event(enable_timing=True, external=graph)) for _ in range(reps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if graph:
        g_each, g_b2b = _graph(fn, reps, evs), _graph(fn, reps)
        g_each.replay()
        t0.record()
        g_b2b.replay()
        t1.record()
    else:
        for e0, e1 in evs:
            e0.record()
            fn()
            e1.record()
        t0.record()
        for _ in range(reps):
            fn()
        t1.record()
    torch.cuda.synchronize()
    ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    med = statistics.median(ms)
    b2b = t0.elapsed_time(t1) / reps
    scale = 1e9 if unit == "B" else 1e12
    return {"op": op, "case": desc, "launch_ms_median": round(med, 5),
            "launch_ms_min": round(min(ms), 5), "launch_ms_max": round(max(ms), 5),
            "back_to_back_ms": round(b2b, 5), "reps": reps, "graph": graph,
            "work": work, "work_unit": unit,
            "rate": round(work / (med / 1e3) / scale, 1),
            "rate_back_to_back": round(work / (b2b / 1e3) / scale, 1),
            "rate_unit": "GB/s" if unit == "B" else "TFLOP/s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", required=True, choices=OPS)
    ap.add_argument("--workload", default="video", choices=sorted(W.WORKLOADS))
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--cols", type=int, default=None, help="RMSNorm width C")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--eager", action="store_true",
                    help="launch from Python one call at a time instead of CUDA graphs")
    a = ap.parse_args()
    if a.cols is not None and a.op != "rmsnorm":
        ap.error("--cols applies to --op rmsnorm only")
    print(json.dumps(run(a.op, a.workload, a.rows, a.reps, a.warmup, not a.eager, a.cols)),
          flush=True)


if __name__ == "__main__":
    main()
