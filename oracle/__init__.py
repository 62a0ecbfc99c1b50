"""CPU oracle for the DiT elementwise hot path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA path: the
arithmetic lives in ``dtrot_oracle.c`` (plain C, IEEE double with explicit
bf16/fp32 rounding), and this module only marshals numpy arrays into it.

bf16 tensors are passed as ``numpy.uint16`` bit patterns; use
``bf16_bits(t)`` / ``from_bits(a)`` to move between torch bf16 tensors and
bit arrays.

Functions and the passages they follow:
  rope_cos_sin       ERNIE-Image fusion page, section 1 (cos/sin once per
                     forward, (B*S, rot_dim) rows, fp32 cos then bf16 cast).
  rope_rotate_half   same page, section 2 (rotate-half, per-op bf16 rounding,
                     round(round(x1*cos1) + round(-x2*sin1)), tail passthrough).
  gelu_and_mul       same page, section 3 (up * gelu(gate), activation rounded
                     to bf16 before the multiply).
  rmsnorm_residual   sequence-parallelism post, per-token RMSNorm and residual
                     add, Pre-Norm order (add, then normalise).
  gate_up_bf16       same ERNIE-Image page, section 3 (the MLP's gate_up
                     projection feeding GEGLU): x W^T rounded to bf16, with
                     bounds for an fp32 accumulation in any order.
  gemm_gelu_and_mul  gate_up_bf16 followed by gelu_and_mul (gate = first F
                     output features).
  *_f64              the same row formulas with every rounding removed, used by
                     the invariant pins (norm preservation, relative position,
                     unit RMS).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None
_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.dto_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.dto_bf16_to_double.restype = ctypes.c_double
        L.dto_rn16.argtypes = [ctypes.c_double]
        L.dto_rn16.restype = ctypes.c_uint16
        L.dto_rn32.argtypes = [ctypes.c_double]
        L.dto_rn32.restype = ctypes.c_float
        L.dto_rn16_of_rn32.argtypes = [ctypes.c_double]
        L.dto_rn16_of_rn32.restype = ctypes.c_uint16
        L.dto_fp_env_ok.argtypes = []
        L.dto_fp_env_ok.restype = ctypes.c_int
        L.dto_gelu_f64.argtypes = [ctypes.c_double]
        L.dto_gelu_f64.restype = ctypes.c_double
        L.dto_gelu_bf16.argtypes = [ctypes.c_uint16]
        L.dto_gelu_bf16.restype = ctypes.c_uint16
        L.dto_rope_cos_sin.argtypes = [_p, _i64, _i64, _i64, _p, _p]
        L.dto_rope_cos_sin.restype = None
        L.dto_rope_cos_sin_f64.argtypes = [_p, _i64, _i64, _i64, _p, _p]
        L.dto_rope_cos_sin_f64.restype = None
        L.dto_rope_rotate_half.argtypes = [_p] + [_i64] * 7 + [_p, _p, _i64, _p] + [_i64] * 3
        L.dto_rope_rotate_half.restype = None
        L.dto_rope_rotate_half_f64.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _p, _i64, _p]
        L.dto_rope_rotate_half_f64.restype = None
        L.dto_gelu_and_mul.argtypes = [_p, _i64, _p, _i64, _p, _i64, _i64, _i64]
        L.dto_gelu_and_mul.restype = None
        L.dto_rmsnorm_residual.argtypes = [_p, _i64, _p, _i64, _p, ctypes.c_double, _p,
                                           _i64, _i64, _i64]
        L.dto_rmsnorm_residual.restype = None
        L.dto_rmsnorm_residual_f64.argtypes = [_p, _p, _p, ctypes.c_double, _p, _p,
                                               _i64, _i64]
        L.dto_rmsnorm_residual_f64.restype = None
        L.dto_gate_up_bf16.argtypes = [_p, _i64, _i64, _p, _i64, ctypes.c_double, _p, _p, _p]
        L.dto_gate_up_bf16.restype = None
        L.dto_set_num_threads.argtypes = [ctypes.c_int]
        L.dto_set_num_threads.restype = None
        L.dto_num_threads.argtypes = []
        L.dto_num_threads.restype = ctypes.c_int
        if not L.dto_fp_env_ok():
            raise RuntimeError("oracle: the FP environment flushes subnormals")
        _LIB = L
    return _LIB


def num_threads() -> int:
    return int(lib().dto_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the row loops use from now on (results do not depend on it)."""
    lib().dto_set_num_threads(int(n))


# ---------------------------------------------------------------- helpers

def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def bf16_bits(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> contiguous numpy uint16 bit array."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray):
    """numpy uint16 bit array -> torch bf16 CPU tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bits_to_f64(a: np.ndarray) -> np.ndarray:
    a = _u16(a)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rn16(v: float) -> int:
    return int(lib().dto_rn16(float(v)))


def rn16_of_rn32(v: float) -> int:
    return int(lib().dto_rn16_of_rn32(float(v)))


def rn32(v: float) -> float:
    return float(lib().dto_rn32(float(v)))


def rn16_array(v: np.ndarray) -> np.ndarray:
    """Vector form of rn16 (a python loop over the C routine; small inputs)."""
    f = lib().dto_rn16
    flat = np.asarray(v, dtype=np.float64).ravel()
    return np.array([f(float(x)) for x in flat], dtype=np.uint16).reshape(np.shape(v))


def gelu_f64(x: float) -> float:
    return float(lib().dto_gelu_f64(float(x)))


def gelu_bf16(xb: int) -> int:
    return int(lib().dto_gelu_bf16(int(xb)))


# ---------------------------------------------------------------- cos/sin tables

def rope_cos_sin(freqs: np.ndarray):
    """freqs fp32 (S, B, 1, R) -> (cos, sin), each uint16 (B*S, R)."""
    f = np.ascontiguousarray(freqs, dtype=np.float32)
    if f.ndim != 4 or f.shape[2] != 1:
        raise ValueError("freqs must be (S, B, 1, R)")
    S, B, _, R = f.shape
    cos = np.empty((B * S, R), dtype=np.uint16)
    sin = np.empty((B * S, R), dtype=np.uint16)
    lib().dto_rope_cos_sin(_ptr(f), S, B, R, _ptr(cos), _ptr(sin))
    return cos, sin


def rope_cos_sin_f64(freqs: np.ndarray):
    f = np.ascontiguousarray(freqs, dtype=np.float64)
    S, B, _, R = f.shape
    cos = np.empty((B * S, R), dtype=np.float64)
    sin = np.empty((B * S, R), dtype=np.float64)
    lib().dto_rope_cos_sin_f64(_ptr(f), S, B, R, _ptr(cos), _ptr(sin))
    return cos, sin


# ---------------------------------------------------------------- RoPE

def rope_rotate_half(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """x uint16 (B, S, H, D) (any element strides, last dim contiguous);
    cos/sin uint16 (B*S, rot) -> out uint16 (B, S, H, D) contiguous."""
    x = _u16(x)
    if x.ndim != 4 or x.strides[3] != 2:
        x = np.ascontiguousarray(x)
    B, S, H, D = x.shape
    cos = np.ascontiguousarray(_u16(cos))
    sin = np.ascontiguousarray(_u16(sin))
    rot = cos.shape[1]
    if cos.shape != (B * S, rot) or sin.shape != cos.shape:
        raise ValueError("cos/sin must be (B*S, rot)")
    if rot % 2 or rot > D or rot <= 0:
        raise ValueError("rot must be even and in (0, D]")
    out = np.empty((B, S, H, D), dtype=np.uint16)
    sx = [st // 2 for st in x.strides[:3]]
    lib().dto_rope_rotate_half(_ptr(x), B, S, H, D, sx[0], sx[1], sx[2], _ptr(cos),
                               _ptr(sin), rot, _ptr(out), S * H * D, H * D, D)
    return out


def rope_rotate_half_f64(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    B, S, H, D = x.shape
    cos = np.ascontiguousarray(cos, dtype=np.float64)
    sin = np.ascontiguousarray(sin, dtype=np.float64)
    rot = cos.shape[1]
    out = np.empty_like(x)
    lib().dto_rope_rotate_half_f64(_ptr(x), B, S, H, D, _ptr(cos), _ptr(sin), rot, _ptr(out))
    return out


# ---------------------------------------------------------------- GEGLU

def gelu_and_mul(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """gate, up uint16 (T, F) (row strides allowed) -> out uint16 (T, F)."""
    gate, up = _u16(gate), _u16(up)
    if gate.shape != up.shape or gate.ndim != 2:
        raise ValueError("gate and up must both be (T, F)")
    if gate.strides[1] != 2:
        gate = np.ascontiguousarray(gate)
    if up.strides[1] != 2:
        up = np.ascontiguousarray(up)
    T, F = gate.shape
    out = np.empty((T, F), dtype=np.uint16)
    lib().dto_gelu_and_mul(_ptr(gate), gate.strides[0] // 2, _ptr(up), up.strides[0] // 2,
                           _ptr(out), F, T, F)
    return out


def gelu_and_mul_fused(gate_up: np.ndarray) -> np.ndarray:
    """(T, 2F) buffer: gate = columns [0, F), up = columns [F, 2F)."""
    gate_up = np.ascontiguousarray(_u16(gate_up))
    F = gate_up.shape[1] // 2
    return gelu_and_mul(gate_up[:, :F], gate_up[:, F:2 * F])


# ---------------------------------------------------------------- RMSNorm + residual

def rmsnorm_residual(x: np.ndarray, residual: np.ndarray, w: np.ndarray, eps: float):
    """x, residual uint16 (T, C); w uint16 (C,) -> (h, y) uint16 (T, C).
    h is the updated residual stream; the input arrays are not modified."""
    x = np.ascontiguousarray(_u16(x))
    h = np.array(_u16(residual), dtype=np.uint16, copy=True, order="C")
    w = np.ascontiguousarray(_u16(w))
    T, C = x.shape
    if h.shape != (T, C) or w.shape != (C,):
        raise ValueError("shapes: x (T, C), residual (T, C), w (C,)")
    y = np.empty((T, C), dtype=np.uint16)
    lib().dto_rmsnorm_residual(_ptr(x), C, _ptr(h), C, _ptr(w), float(eps), _ptr(y), C, T, C)
    return h, y


def rmsnorm_residual_f64(x, residual, w, eps):
    x = np.ascontiguousarray(x, dtype=np.float64)
    r = np.ascontiguousarray(residual, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    T, C = x.shape
    h = np.empty_like(x)
    y = np.empty_like(x)
    lib().dto_rmsnorm_residual_f64(_ptr(x), _ptr(r), _ptr(w), float(eps), _ptr(h), _ptr(y),
                                   T, C)
    return h, y


# ---------------------------------------------------------------- gate_up projection + GEGLU

def gate_up_bf16(x: np.ndarray, w: np.ndarray, eps: float = 0.0):
    """x uint16 (T, C), w uint16 (N, C) -> (exact, lo, hi) uint16 (T, N): the
    bf16 rounding of x W^T, and the roundings of its ends when each dot product
    may be off by eps * sum|x w| (an fp32 accumulation in any order)."""
    x = np.ascontiguousarray(_u16(x))
    w = np.ascontiguousarray(_u16(w))
    T, C = x.shape
    N = w.shape[0]
    if w.shape[1] != C:
        raise ValueError("x is (T, C) and w is (N, C)")
    exact = np.empty((T, N), dtype=np.uint16)
    lo = np.empty((T, N), dtype=np.uint16)
    hi = np.empty((T, N), dtype=np.uint16)
    lib().dto_gate_up_bf16(_ptr(x), T, C, _ptr(w), N, float(eps), _ptr(exact), _ptr(lo),
                           _ptr(hi))
    return exact, lo, hi


def gemm_gelu_and_mul(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """GEGLU of the bf16 gate_up projection: w (2F, C), gate rows first."""
    gu, _, _ = gate_up_bf16(x, w)
    F = w.shape[0] // 2
    return gelu_and_mul(gu[:, :F], gu[:, F:])
