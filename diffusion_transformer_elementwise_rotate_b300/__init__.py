"""B300-native elementwise hot path of a diffusion-transformer block.

Four ops, each one sm_103a CUDA kernel behind the C ABI in include/dtrot.h:
rotary cos/sin tables, rotate-half RoPE, GEGLU with activation rounding, and
RMSNorm fused with the residual add.  The torch wrappers in `api` only pass
pointers, sizes and strides; `_capi` is the raw ctypes binding.
"""
from . import selfcheck  # noqa: F401
from ._capi import DtrotError, DtrotKernelError, DtrotUnavailable, load  # noqa: F401
from .api import (gelu_and_mul, gelu_and_mul_fused, gelu_table, gelu_table_build,  # noqa: F401
                  gelu_workspace, gemm_error_word, gemm_gelu_and_mul,
                  rmsnorm_residual, rope_cos_sin_precompute, rope_rotate_half,
                  rope_rotate_half_qk, rope_rotate_half_qk_)
