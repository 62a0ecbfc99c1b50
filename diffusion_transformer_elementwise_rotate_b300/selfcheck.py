"""Opt-in first-call self-check of the fused ops against plain PyTorch on the GPU.

The ERNIE-Image fusion page ("why this is good", item 2, and the review-feedback
section) describes a gate that, on the first call for a given shape, dtype and
platform, compares the fused op with the eager PyTorch chain using
torch.equal.  Here the same check is opt-in (enable() or DTROT_SELF_CHECK=1)
and, since nothing here falls back to another implementation, a mismatch
raises SelfCheckError instead of switching paths.

References (plain torch ops on the same device and stream):
  RoPE     the eager bf16 chunk / neg / cat / mul / add chain: must be equal
           bit for bit (NaN payloads aside).
  tables   torch.cos / torch.sin in fp64, rounded to fp32 and then to bf16.
  GEGLU    gelu in fp64 (as x/2 * erfc(-x/sqrt 2), which keeps its relative
           accuracy for x << 0), rounded to fp32 and then bf16, times up.
  RMSNorm  h = x + r in bf16 (bit for bit), then the norm in fp64.
The last three must agree within 1 bf16 ulp on every element, with at most
0.01% of the elements different (the fp64 references can still differ from
the exactly rounded result in rounding-tie corner cases).  GEGLU after the
gate_up projection is compared with the fp64 projection rounded to bf16 and
the projection is checked on its first 256 rows, which the kernel runs again
with the rounded gate_up stored: the rerun must give the same output bits,
the output must be the GEGLU reference of the stored gate and up (the
tolerance above), and every stored gate and up must lie within the bf16
rounding of the fp64 projection widened by the fp32 accumulation bound
(C + 1) * 2^-23 * sum|x w| (the tensor cores sum in fp32 in their own order,
so near-cancelling sums can move by several bf16 steps).

The check costs a synchronisation and temporary tensors; it is meant for
bring-up on a new platform or build, not for production steps.
"""
from __future__ import annotations

import os
import threading

import torch

_lock = threading.Lock()
_enabled = os.environ.get("DTROT_SELF_CHECK", "") not in ("", "0")
_seen: set = set()

MAX_ULP = 1
MAX_MISMATCH_FRACTION = 1e-4


class SelfCheckError(RuntimeError):
    pass


def enable() -> None:
    global _enabled
    _enabled = True


def disable() -> None:
    global _enabled
    _enabled = False


def enabled() -> bool:
    return _enabled


def reset() -> None:
    """Forget which (op, shape, device) keys were checked."""
    with _lock:
        _seen.clear()


def checked() -> set:
    with _lock:
        return set(_seen)


def want(op: str, *tensors) -> tuple | None:
    """The key of this call if it is the first one to be checked, else None."""
    if not _enabled:
        return None
    key = (op,) + tuple((tuple(t.shape), t.dtype, str(t.device)) for t in tensors
                        if isinstance(t, torch.Tensor))
    with _lock:
        if key in _seen:
            return None
        _seen.add(key)
    return key


# ---------------------------------------------------------------- comparison

def _ordered(u: torch.Tensor) -> torch.Tensor:
    """bf16 bit patterns (int32) -> integers ordered like the values, with
    +0 and -0 mapped to the same key."""
    mag = u & 0x7FFF
    key = torch.where((u & 0x8000) != 0, 0x8000 - mag, 0x8000 + mag)
    return torch.where(mag == 0, torch.full_like(key, 0x8000), key)


def _is_nan(u: torch.Tensor) -> torch.Tensor:
    return ((u & 0x7F80) == 0x7F80) & ((u & 0x007F) != 0)


def compare(name: str, got: torch.Tensor, ref: torch.Tensor, exact: bool,
            max_fraction: float = MAX_MISMATCH_FRACTION) -> int:
    """Raise SelfCheckError unless `got` matches `ref` (both bf16): bit for bit
    when `exact`, else within MAX_ULP on every element and in at most
    MAX_MISMATCH_FRACTION of them.  Returns the number of differing elements."""
    if got.shape != ref.shape:
        raise SelfCheckError(f"{name}: shape {tuple(got.shape)} != {tuple(ref.shape)}")
    a = got.detach().contiguous().view(torch.int16).to(torch.int32) & 0xFFFF
    b = ref.detach().contiguous().view(torch.int16).to(torch.int32) & 0xFFFF
    both_nan = _is_nan(a) & _is_nan(b)
    one_nan = _is_nan(a) ^ _is_nan(b)
    d = (_ordered(a) - _ordered(b)).abs()
    d = torch.where(both_nan, torch.zeros_like(d), d)
    d = torch.where(one_nan, torch.full_like(d, 1 << 20), d)
    n = int((d != 0).sum().item())
    worst = int(d.max().item()) if d.numel() else 0
    if exact and n:
        raise SelfCheckError(f"{name}: {n} of {d.numel()} elements differ from the eager "
                             f"chain (largest difference {worst} bf16 steps)")
    if not exact and (worst > MAX_ULP or n > max_fraction * d.numel()):
        raise SelfCheckError(f"{name}: {n} of {d.numel()} elements differ, largest difference "
                             f"{worst} bf16 steps")
    return n


# ---------------------------------------------------------------- references

def ref_rope(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor) -> torch.Tensor:
    """The eager bf16 chain: x_rot * cos + cat(-x2, x1) * sin, tail appended."""
    B, S, H, D = x.shape
    rot = cos.shape[1]
    c = cos.view(B, S, 1, rot)
    s = sin.view(B, S, 1, rot)
    xr = x[..., :rot]
    x1, x2 = xr.chunk(2, dim=-1)
    rotated = torch.cat((-x2, x1), dim=-1)
    o = xr * c + rotated * s
    return torch.cat((o, x[..., rot:]), dim=-1)


def ref_tables(freqs: torch.Tensor):
    S, B, _, R = freqs.shape
    f = freqs.permute(1, 0, 2, 3).reshape(B * S, R).double()
    return (torch.cos(f).float().to(torch.bfloat16), torch.sin(f).float().to(torch.bfloat16))


def ref_geglu(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    x = gate.double()
    g = (0.5 * x * torch.special.erfc(-x * 0.7071067811865476)).float().to(torch.bfloat16)
    return (up.float() * g.float()).to(torch.bfloat16)


def ref_rmsnorm(x: torch.Tensor, r: torch.Tensor, w: torch.Tensor, eps: float):
    h = x + r
    hd = h.double()
    eps32 = float(torch.tensor(eps, dtype=torch.float32))  # the kernels take eps as fp32
    inv = torch.rsqrt(hd.pow(2).mean(dim=-1, keepdim=True) + eps32)
    return h, (hd * inv * w.double()).float().to(torch.bfloat16)


def check_gemm_geglu(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor, rerun) -> None:
    """GEGLU after the gate_up projection, on a sample of rows.  `rerun(rows)`
    runs the kernel on x[:rows] and returns (out, gate_up) for them."""
    T, C = x.shape
    F = w.shape[0] // 2
    rows = min(T, 256)
    out_s, gu = rerun(rows)
    compare("gemm_gelu_and_mul rerun", out_s, out[:rows], exact=True)
    compare("gemm_gelu_and_mul epilogue", out[:rows], ref_geglu(gu[:, :F], gu[:, F:]), exact=False)
    xd, wd = x[:rows].double(), w.double()
    dot = xd @ wd.t()
    mag = xd.abs() @ wd.abs().t()
    eps = (C + 1) * 2.0 ** -23
    lo = _ordered((dot - eps * mag).float().to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF)
    hi = _ordered((dot + eps * mag).float().to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF)
    k = _ordered(gu.contiguous().view(torch.int16).to(torch.int32) & 0xFFFF)
    bad = int(((k < lo - 1) | (k > hi + 1)).sum().item())
    if bad:
        raise SelfCheckError(f"gemm_gelu_and_mul: {bad} gate/up values outside the fp32 "
                             "accumulation bounds of the projection")
