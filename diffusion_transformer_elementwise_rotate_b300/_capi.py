"""ctypes binding of libdtrot.so (declarations in include/dtrot.h).

Loading is lazy; if the shared library is missing or cannot be loaded, every
call raises DtrotUnavailable.  There is no fallback: the kernels in libdtrot
are the only implementation of these ops.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdtrot.so")

STATUS = {
    0: "DTROT_OK",
    1: "DTROT_ERR_NULL",
    2: "DTROT_ERR_SHAPE",
    3: "DTROT_ERR_ROTDIM",
    4: "DTROT_ERR_STRIDE",
    5: "DTROT_ERR_ALIAS",
    6: "DTROT_ERR_LAUNCH",
    7: "DTROT_ERR_DEVICE",
    8: "DTROT_ERR_VALUE",
    9: "DTROT_ERR_WORKSPACE",
    10: "DTROT_ERR_ALIGN",
}
OK, ERR_NULL, ERR_SHAPE, ERR_ROTDIM, ERR_STRIDE, ERR_ALIAS, ERR_LAUNCH, ERR_DEVICE, \
    ERR_VALUE, ERR_WORKSPACE, ERR_ALIGN = range(11)

# entry point -> (restype, argtypes); must match include/dtrot.h
_i64 = ctypes.c_int64
_p = ctypes.c_void_p
SIGNATURES = {
    "dtrot_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "dtrot_version": (ctypes.c_int, []),
    "dtrot_rope_cos_sin_precompute": (ctypes.c_int, [_p, _i64, _i64, _i64, _p, _p, _p]),
    "dtrot_rope_rotate_half": (ctypes.c_int,
                               [_p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p, _p, _i64,
                                _p, _i64, _i64, _i64, _p]),
    "dtrot_rope_rotate_half_qk": (ctypes.c_int, [_p, _i64, _i64, _i64, _i64, _p, _i64, _i64,
                                                  _i64, _i64, _i64, _i64, _i64, _p, _p, _p,
                                                  _i64, _p]),
    "dtrot_rope_rotate_half_qk_out": (ctypes.c_int, [_p, _i64, _i64, _i64, _i64, _p, _i64,
                                                      _i64, _i64, _i64, _i64, _i64, _i64, _p,
                                                      _p, _p, _i64, _p, _i64, _i64, _i64, _p,
                                                      _i64, _i64, _i64, _p]),
    "dtrot_gelu_and_mul_workspace_bytes": (ctypes.c_int64, []),
    "dtrot_gelu_and_mul": (ctypes.c_int, [_p, _i64, _p, _i64, _p, _i64, _i64, _i64, _p, _i64,
                                          _p]),
    "dtrot_gelu_table_build": (ctypes.c_int, [_p, _i64, _p]),
    "dtrot_gelu_and_mul_with_table": (ctypes.c_int, [_p, _i64, _p, _i64, _p, _i64, _i64, _i64,
                                                     _p, _i64, _p]),
    "dtrot_gemm_gelu_and_mul_workspace_bytes": (ctypes.c_int64, []),
    "dtrot_gemm_gelu_and_mul": (ctypes.c_int, [_p, _i64, _i64, _p, _i64, _p, _i64, _p, _i64,
                                               _p, _i64, _p]),
    "dtrot_gemm_gelu_and_mul_withhold_last_stage": (ctypes.c_int, [_p, _i64, _i64, _p, _i64, _p,
                                                                   _i64, _p, _i64, _p, _i64,
                                                                   _p]),
    "dtrot_gemm_gelu_and_mul_error": (ctypes.c_int, [_p, _p, _p]),
    "dtrot_gelu_and_mul_noalloc": (ctypes.c_int, [_p, _i64, _p, _i64, _p, _i64, _i64, _i64, _p]),
    "dtrot_rmsnorm_residual": (ctypes.c_int,
                               [_p, _i64, _p, _i64, _p, ctypes.c_float, _p, _i64, _i64, _i64,
                                _p]),
}


class DtrotUnavailable(RuntimeError):
    pass


class DtrotKernelError(RuntimeError):
    """A kernel reported a failure through its error word (its output is not
    valid)."""


class DtrotError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {STATUS.get(code, code)}")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libdtrot.so once; raise DtrotUnavailable if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise DtrotUnavailable(
                    f"{path} is missing; build it with "
                    "`python -m diffusion_transformer_elementwise_rotate_b300.build`")
            try:
                lib = ctypes.CDLL(path)
            except OSError as e:
                raise DtrotUnavailable(f"cannot load {path}: {e}") from e
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def call(name: str, *args) -> int:
    """Call an entry point; returns its dtrot_status code."""
    return int(getattr(load(), name)(*args))


def check(name: str, *args) -> None:
    code = call(name, *args)
    if code != OK:
        raise DtrotError(name, code)
