"""The C ABI boundary, on the host (no GPU needed).

- libdtrot.so loads and exports every entry point include/dtrot.h declares;
- every invalid argument returns its own status code before anything is
  launched (the pointers used here are never dereferenced);
- zero-sized calls are no-ops that return DTROT_OK.
"""
import ctypes
import os
import re

import pytest
import torch

from diffusion_transformer_elementwise_rotate_b300 import _capi
from diffusion_transformer_elementwise_rotate_b300 import build as dbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dtrot.h")


# Calls whose arguments pass validation go on to the launch.  With the fake
# pointers used here they may only run where no CUDA device is visible (they
# then return DTROT_ERR_DEVICE): on a machine with a GPU they would launch
# kernels on unmapped addresses, so those tests are skipped there.
no_device = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="valid calls on fake pointers would launch on the GPU")


@pytest.fixture(scope="module")
def lib():
    dbuild.build()
    return _capi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dtrot_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_ops():
    names = declared_functions()
    for op in ("dtrot_rope_cos_sin_precompute", "dtrot_rope_rotate_half",
               "dtrot_rope_rotate_half_qk", "dtrot_rope_rotate_half_qk_out",
               "dtrot_gelu_and_mul",
               "dtrot_gelu_and_mul_workspace_bytes", "dtrot_gelu_table_build",
               "dtrot_gelu_and_mul_with_table", "dtrot_gemm_gelu_and_mul",
               "dtrot_gemm_gelu_and_mul_workspace_bytes", "dtrot_gemm_gelu_and_mul_error",
               "dtrot_gemm_gelu_and_mul_withhold_last_stage", "dtrot_gelu_and_mul_noalloc",
               "dtrot_rmsnorm_residual",
               "dtrot_status_str", "dtrot_version"):
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _capi.SIGNATURES, f"{name} has no ctypes signature"


def test_status_strings(lib):
    for code, name in _capi.STATUS.items():
        s = lib.dtrot_status_str(code).decode()
        assert s.startswith(name)
    assert lib.dtrot_version() >= 200


P = 0x100000  # fake, 256-byte aligned device addresses (never dereferenced)
Q = 0x900000
R = 0x1100000
W = 0x1900000


def rope(**kw):
    a = dict(x=P, B=1, S=4, H=2, D=8, sx_b=64, sx_s=16, sx_h=8, cos=Q, sin=R, rot=8, out=W,
             so_b=64, so_s=16, so_h=8)
    a.update(kw)
    return _capi.call("dtrot_rope_rotate_half", a["x"], a["B"], a["S"], a["H"], a["D"],
                      a["sx_b"], a["sx_s"], a["sx_h"], a["cos"], a["sin"], a["rot"], a["out"],
                      a["so_b"], a["so_s"], a["so_h"], None)


WS = 0x2100000   # fake workspace
WS_BYTES = 131072


def geglu(**kw):
    a = dict(gate=P, sg=16, up=P + 16, su=16, out=W, so=8, T=4, F=8, ws=WS, wsb=WS_BYTES)
    a.update(kw)
    return _capi.call("dtrot_gelu_and_mul", a["gate"], a["sg"], a["up"], a["su"], a["out"],
                      a["so"], a["T"], a["F"], a["ws"], a["wsb"], None)


def rms(**kw):
    a = dict(x=P, sx=8, res=Q, sr=8, w=R, eps=1e-6, out=W, so=8, T=4, C=8)
    a.update(kw)
    return _capi.call("dtrot_rmsnorm_residual", a["x"], a["sx"], a["res"], a["sr"], a["w"],
                      a["eps"], a["out"], a["so"], a["T"], a["C"], None)


def tables(**kw):
    a = dict(f=P, S=4, B=2, R=8, c=Q, s=R)
    a.update(kw)
    return _capi.call("dtrot_rope_cos_sin_precompute", a["f"], a["S"], a["B"], a["R"], a["c"],
                      a["s"], None)


def rope_qk(**kw):
    # q heads [0, 2) and k heads [2, 4) of one (1, 4, 6, 8) QKV buffer at P
    a = dict(q=P, Hq=2, sq_b=192, sq_s=48, sq_h=8, k=P + 2 * 16, Hk=2, sk_b=192, sk_s=48, sk_h=8,
             B=1, S=4, D=8, cos=Q, sin=R, freqs=0, rot=8)
    a.update(kw)
    return _capi.call("dtrot_rope_rotate_half_qk", a["q"], a["Hq"], a["sq_b"], a["sq_s"],
                      a["sq_h"], a["k"], a["Hk"], a["sk_b"], a["sk_s"], a["sk_h"], a["B"],
                      a["S"], a["D"], a["cos"] or None, a["sin"] or None, a["freqs"] or None,
                      a["rot"], None)


def test_rope_qk_validation(lib):
    assert rope_qk(S=0, q=0, k=0, cos=0, sin=0) == _capi.OK
    assert rope_qk(Hq=0, Hk=0) == _capi.OK
    assert rope_qk(q=0) == _capi.ERR_NULL
    assert rope_qk(cos=0) == _capi.ERR_NULL
    assert rope_qk(freqs=W) == _capi.ERR_VALUE                        # tables and angles
    assert rope_qk(rot=6, D=4) == _capi.ERR_ROTDIM
    assert rope_qk(rot=5) == _capi.ERR_ROTDIM
    assert rope_qk(Hk=-1) == _capi.ERR_SHAPE
    assert rope_qk(sq_h=0) == _capi.ERR_STRIDE
    assert rope_qk(sk_h=4) == _capi.ERR_STRIDE                        # k rows overlap
    assert rope_qk(k=P + 2 * 8) == _capi.ERR_ALIAS                    # k starts inside q
    assert rope_qk(k=P + 2 * 16, sk_s=96) == _capi.ERR_ALIAS          # interleaved, other strides
    assert rope_qk(cos=P) == _capi.ERR_ALIAS                          # tables over q
    assert rope_qk(cos=0, sin=0, freqs=P + 2 * 40) == _capi.ERR_ALIAS  # angles over k


@pytest.mark.skipif(torch.cuda.is_available(), reason="host without a GPU only")
@no_device
def test_rope_qk_valid_layouts_reach_the_device_check(lib):
    assert rope_qk(Hq=0, q=0, k=P) == _capi.ERR_DEVICE                 # k alone
    assert rope_qk() == _capi.ERR_DEVICE                               # fused QKV slices
    assert rope_qk(q=P + 2 * 16, k=P) == _capi.ERR_DEVICE              # k heads before q heads
    assert rope_qk(k=W, sk_b=64, sk_s=16) == _capi.ERR_DEVICE          # separate buffers
    assert rope_qk(cos=0, sin=0, freqs=Q) == _capi.ERR_DEVICE          # angles


def rope_qk_out(**kw):
    # q heads [0, 2) and k heads [2, 4) of one (1, 4, 6, 8) QKV buffer at P,
    # rotated into the two head ranges of one (1, 4, 4, 8) buffer at W
    a = dict(q=P, Hq=2, sq_b=192, sq_s=48, sq_h=8, k=P + 2 * 16, Hk=2, sk_b=192, sk_s=48, sk_h=8,
             B=1, S=4, D=8, cos=Q, sin=R, freqs=0, rot=8,
             qo=W, soq_b=128, soq_s=32, soq_h=8, ko=W + 2 * 16, sok_b=128, sok_s=32, sok_h=8)
    a.update(kw)
    return _capi.call("dtrot_rope_rotate_half_qk_out", a["q"] or None, a["Hq"], a["sq_b"],
                      a["sq_s"], a["sq_h"], a["k"] or None, a["Hk"], a["sk_b"], a["sk_s"],
                      a["sk_h"], a["B"], a["S"], a["D"], a["cos"] or None, a["sin"] or None,
                      a["freqs"] or None, a["rot"], a["qo"] or None, a["soq_b"], a["soq_s"],
                      a["soq_h"], a["ko"] or None, a["sok_b"], a["sok_s"], a["sok_h"], None)


def test_rope_qk_out_validation(lib):
    assert rope_qk_out(S=0, q=0, k=0, cos=0, sin=0, qo=0, ko=0) == _capi.OK
    assert rope_qk_out(Hq=0, Hk=0) == _capi.OK
    assert rope_qk_out(q=0) == _capi.ERR_NULL
    assert rope_qk_out(ko=0) == _capi.ERR_NULL
    assert rope_qk_out(sin=0) == _capi.ERR_NULL
    assert rope_qk_out(freqs=WS) == _capi.ERR_VALUE                    # tables and angles
    assert rope_qk_out(rot=10) == _capi.ERR_ROTDIM
    assert rope_qk_out(Hq=-2) == _capi.ERR_SHAPE
    assert rope_qk_out(sq_s=0) == _capi.ERR_STRIDE                     # input stride 0
    assert rope_qk_out(soq_h=0) == _capi.ERR_STRIDE
    assert rope_qk_out(sok_h=4) == _capi.ERR_STRIDE                    # k_out rows overlap
    assert rope_qk_out(ko=W + 2 * 8) == _capi.ERR_ALIAS                # k_out inside q_out
    assert rope_qk_out(ko=W + 2 * 16, sok_s=64) == _capi.ERR_ALIAS     # interleaved, other strides
    assert rope_qk_out(qo=P) == _capi.ERR_ALIAS                        # output over q
    assert rope_qk_out(ko=P + 2 * 32, sok_b=192, sok_s=48) == _capi.ERR_ALIAS  # over q's span
    assert rope_qk_out(cos=W + 2 * 40) == _capi.ERR_ALIAS              # tables under k_out
    assert rope_qk_out(cos=0, sin=0, freqs=W) == _capi.ERR_ALIAS       # angles under q_out


@pytest.mark.skipif(torch.cuda.is_available(), reason="host without a GPU only")
@no_device
def test_rope_qk_out_valid_layouts_reach_the_device_check(lib):
    assert rope_qk_out() == _capi.ERR_DEVICE                            # fused in, fused out
    assert rope_qk_out(k=P) == _capi.ERR_DEVICE                         # inputs may overlap
    assert rope_qk_out(Hk=0, k=0, ko=0) == _capi.ERR_DEVICE             # q alone
    assert rope_qk_out(ko=R + 4096, sok_b=64, sok_s=16) == _capi.ERR_DEVICE  # separate outputs
    assert rope_qk_out(cos=0, sin=0, freqs=Q) == _capi.ERR_DEVICE       # angles


def gemm(**kw):
    a = dict(x=P, T=4, C=64, w=Q, F=16, out=R, so=16, gu=0, sgu=32, ws=WS, wsb=17408)
    a.update(kw)
    return _capi.call("dtrot_gemm_gelu_and_mul", a["x"], a["T"], a["C"], a["w"], a["F"],
                      a["out"], a["so"], a["gu"] or None, a["sgu"], a["ws"], a["wsb"], None)


def test_gemm_gelu_and_mul_validation(lib):
    assert lib.dtrot_gemm_gelu_and_mul_workspace_bytes() == 17408
    assert gemm(T=0, x=0, w=0, out=0, ws=0) == _capi.OK
    assert gemm(F=0) == _capi.OK
    assert gemm(C=0) == _capi.ERR_SHAPE
    assert gemm(T=-1) == _capi.ERR_SHAPE
    assert gemm(T=1 << 31) == _capi.ERR_SHAPE
    assert gemm(w=0) == _capi.ERR_NULL
    assert gemm(ws=0) == _capi.ERR_NULL
    assert gemm(so=8) == _capi.ERR_STRIDE                  # < F
    assert gemm(C=60) == _capi.ERR_ALIGN
    assert gemm(F=12, so=16) == _capi.ERR_ALIGN
    assert gemm(x=P + 8) == _capi.ERR_ALIGN
    assert gemm(so=20) == _capi.ERR_ALIGN
    assert gemm(wsb=17407) == _capi.ERR_WORKSPACE
    assert gemm(ws=WS + 4) == _capi.ERR_WORKSPACE
    assert gemm(out=P) == _capi.ERR_ALIAS                  # over x
    assert gemm(ws=Q + 64) == _capi.ERR_ALIAS              # over w
    assert gemm(gu=W, sgu=16) == _capi.ERR_STRIDE          # < 2F
    assert gemm(gu=W + 8) == _capi.ERR_ALIGN
    assert gemm(gu=R + 32) == _capi.ERR_ALIAS              # over out


@pytest.mark.skipif(torch.cuda.is_available(), reason="host without a GPU only")
@no_device
def test_gemm_gelu_and_mul_valid_call_reaches_device_check(lib):
    assert gemm() == _capi.ERR_DEVICE
    assert gemm(gu=W) == _capi.ERR_DEVICE
    assert _capi.call("dtrot_gemm_gelu_and_mul_withhold_last_stage", P, 4, 64, Q, 16, R, 16,
                      None, 32, WS, 17408, None) == _capi.ERR_DEVICE
    word = ctypes.c_uint32(0)
    assert _capi.call("dtrot_gemm_gelu_and_mul_error", WS, ctypes.addressof(word),
                      None) == _capi.ERR_DEVICE


def test_gemm_error_word_read_validation(lib):
    word = ctypes.c_uint32(0)
    assert _capi.call("dtrot_gemm_gelu_and_mul_error", None, ctypes.addressof(word),
                      None) == _capi.ERR_NULL
    assert _capi.call("dtrot_gemm_gelu_and_mul_error", WS, None, None) == _capi.ERR_NULL
    assert _capi.call("dtrot_gemm_gelu_and_mul_error", WS + 4, ctypes.addressof(word),
                      None) == _capi.ERR_WORKSPACE
    # the diagnostic run validates like the plain call
    assert _capi.call("dtrot_gemm_gelu_and_mul_withhold_last_stage", P, 4, 60, Q, 16, R, 16,
                      None, 32, WS, 17408, None) == _capi.ERR_ALIGN


def test_zero_sized_calls_are_noops(lib):
    assert rope(B=0, x=0, cos=0, sin=0, out=0) == _capi.OK
    assert rope(H=0) == _capi.OK
    assert geglu(T=0, gate=0, up=0, out=0) == _capi.OK
    assert rms(C=0, x=0, res=0, w=0, out=0) == _capi.OK
    assert tables(S=0, f=0, c=0, s=0) == _capi.OK
    assert rope_qk_out(B=0, q=0, k=0, cos=0, sin=0, qo=0, ko=0) == _capi.OK


def test_null_pointers(lib):
    assert rope(x=0) == _capi.ERR_NULL
    assert rope(cos=0) == _capi.ERR_NULL
    assert rope(out=0) == _capi.ERR_NULL
    assert geglu(up=0) == _capi.ERR_NULL
    assert geglu(ws=0) == _capi.ERR_NULL
    assert rms(w=0) == _capi.ERR_NULL
    assert tables(s=0) == _capi.ERR_NULL


def test_negative_and_overflowing_sizes(lib):
    assert rope(S=-1) == _capi.ERR_SHAPE
    assert rope(B=1 << 40, S=1 << 40) == _capi.ERR_SHAPE
    assert geglu(F=-8) == _capi.ERR_SHAPE
    assert geglu(T=1 << 62, F=1 << 2) == _capi.ERR_SHAPE
    assert rms(T=-3) == _capi.ERR_SHAPE
    assert tables(R=-2) == _capi.ERR_SHAPE


def test_rot_dim(lib):
    assert rope(rot=7) == _capi.ERR_ROTDIM
    assert rope(rot=0) == _capi.ERR_ROTDIM
    assert rope(rot=10) == _capi.ERR_ROTDIM  # > D
    assert rope(rot=-2) == _capi.ERR_ROTDIM


@no_device
def test_workspace_in_the_gap_between_rows_is_allowed(lib):
    sg = 2 * 65536 + 64
    assert geglu(sg=sg, su=sg, up=P + 16, ws=P + 2 * 32) == _capi.ERR_DEVICE


@no_device
def test_output_strides_in_any_dimension_order(lib):
    # heads outermost, then batch, then tokens: no two elements of out meet
    assert rope(B=2, sx_b=64, so_h=64, so_b=32, so_s=8) == _capi.ERR_DEVICE
    # the same order with token rows 4 elements apart: rows overlap
    assert rope(B=2, sx_b=64, so_h=64, so_b=32, so_s=4) == _capi.ERR_STRIDE
    # heads 16 apart inside a token span of 31 elements: overlap
    assert rope(B=2, sx_b=64, so_h=16, so_b=64, so_s=8) == _capi.ERR_STRIDE


def test_strides(lib):
    assert rope(sx_h=0) == _capi.ERR_STRIDE
    assert rope(so_h=4) == _capi.ERR_STRIDE          # output heads overlap
    assert rope(so_b=0, B=2) == _capi.ERR_STRIDE
    assert geglu(sg=4) == _capi.ERR_STRIDE          # < F
    assert geglu(so=7) == _capi.ERR_STRIDE
    assert rms(sr=7) == _capi.ERR_STRIDE


def test_aliasing(lib):
    # out overlapping x but not identical
    assert rope(out=P + 2) == _capi.ERR_ALIAS
    # in place with different strides
    assert rope(out=P, so_b=128, so_s=32, so_h=16, B=1) == _capi.ERR_ALIAS
    # out overlapping the tables
    assert rope(out=Q) == _capi.ERR_ALIAS
    # GEGLU out over up
    assert geglu(out=P + 16, so=16) == _capi.ERR_ALIAS
    # out partially over gate
    assert geglu(out=P + 8, so=16) == _capi.ERR_ALIAS
    # RMSNorm: out over x / residual / w; x partly over residual; w inside residual rows
    assert rms(out=P) == _capi.ERR_ALIAS
    assert rms(out=Q) == _capi.ERR_ALIAS
    assert rms(out=R) == _capi.ERR_ALIAS
    assert rms(x=Q + 2) == _capi.ERR_ALIAS
    assert rms(w=Q + 8) == _capi.ERR_ALIAS
    # tables: cos and sin overlap
    assert tables(s=Q + 2) == _capi.ERR_ALIAS
    assert tables(c=P) == _capi.ERR_ALIAS


def test_gelu_workspace(lib):
    assert lib.dtrot_gelu_and_mul_workspace_bytes() == WS_BYTES
    assert geglu(wsb=WS_BYTES - 1) == _capi.ERR_WORKSPACE
    assert geglu(wsb=0) == _capi.ERR_WORKSPACE
    assert geglu(ws=WS + 8) == _capi.ERR_WORKSPACE            # not 16-byte aligned
    assert geglu(ws=P) == _capi.ERR_ALIAS                      # over gate
    assert geglu(ws=W - 64) == _capi.ERR_ALIAS                 # runs into out
    sg = 2 * 65536 + 64
    # starts in the gap between two long rows of gate/up but runs into row 1 of gate (element sg)
    assert geglu(sg=sg, su=sg, up=P + 16, ws=P + 2 * (sg - 65536 + 8)) == _capi.ERR_ALIAS
    assert geglu(sg=sg, su=sg, up=P + 16, ws=P + 2 * sg) == _capi.ERR_ALIAS


def geglu_tab(**kw):
    a = dict(gate=P, sg=16, up=P + 16, su=16, out=W, so=8, T=4, F=8, tab=WS, tb=WS_BYTES)
    a.update(kw)
    return _capi.call("dtrot_gelu_and_mul_with_table", a["gate"], a["sg"], a["up"], a["su"],
                      a["out"], a["so"], a["T"], a["F"], a["tab"], a["tb"], None)


def test_prebuilt_gelu_table_validation(lib):
    assert _capi.call("dtrot_gelu_table_build", None, WS_BYTES, None) == _capi.ERR_NULL
    assert _capi.call("dtrot_gelu_table_build", WS, WS_BYTES - 2, None) == _capi.ERR_WORKSPACE
    assert _capi.call("dtrot_gelu_table_build", WS + 8, WS_BYTES, None) == _capi.ERR_WORKSPACE
    assert geglu_tab(T=0, gate=0, up=0, out=0, tab=0) == _capi.OK
    assert geglu_tab(tab=0) == _capi.ERR_NULL
    assert geglu_tab(tb=100) == _capi.ERR_WORKSPACE
    assert geglu_tab(tab=WS + 4) == _capi.ERR_WORKSPACE
    assert geglu_tab(sg=4) == _capi.ERR_STRIDE
    assert geglu_tab(out=P + 16, so=16) == _capi.ERR_ALIAS          # out over up
    assert geglu_tab(tab=W - 64) == _capi.ERR_ALIAS                 # table runs into out


@pytest.mark.skipif(torch.cuda.is_available(), reason="host without a GPU only")
@no_device
def test_prebuilt_gelu_table_valid_calls_reach_device_check(lib):
    assert _capi.call("dtrot_gelu_table_build", WS, WS_BYTES, None) == _capi.ERR_DEVICE
    assert geglu_tab() == _capi.ERR_DEVICE
    assert geglu_tab(tab=P) == _capi.ERR_DEVICE                     # table over gate: both read


def test_eps(lib):
    assert rms(eps=-1.0) == _capi.ERR_VALUE
    assert rms(eps=float("nan")) == _capi.ERR_VALUE
    assert rms(eps=float("inf")) == _capi.ERR_VALUE


@pytest.mark.skipif(torch.cuda.is_available(), reason="host without a GPU only")
@no_device
def test_valid_calls_report_missing_device(lib):
    # arguments that pass validation reach the device check, which fails here
    assert rope() == _capi.ERR_DEVICE
    assert rope(out=P) == _capi.ERR_DEVICE          # in place is valid
    assert geglu() == _capi.ERR_DEVICE              # gate/up halves of one buffer
    assert geglu(out=P, so=16) == _capi.ERR_DEVICE  # out == gate in place
    assert rms() == _capi.ERR_DEVICE
    assert rms(x=Q, sx=8) == _capi.ERR_DEVICE       # x == residual
    assert tables() == _capi.ERR_DEVICE


def test_missing_library_fails_loudly(tmp_path):
    saved = _capi._lib
    _capi._lib = None
    try:
        with pytest.raises(_capi.DtrotUnavailable):
            _capi.load(str(tmp_path / "missing.so"))
    finally:
        _capi._lib = saved


def geglu_noalloc(**kw):
    a = dict(gate=P, sg=16, up=P + 16, su=16, out=W, so=8, T=4, F=8)
    a.update(kw)
    return _capi.call("dtrot_gelu_and_mul_noalloc", a["gate"], a["sg"], a["up"], a["su"],
                      a["out"], a["so"], a["T"], a["F"], None)


def test_noalloc_gelu_and_mul_rejects_what_the_workspace_entry_point_rejects(lib):
    # every invalid call returns its status before the device is queried, and
    # the same status as dtrot_gelu_and_mul with a valid workspace
    cases = [dict(T=-1), dict(F=-8), dict(T=1 << 62, F=4), dict(gate=0), dict(up=0),
             dict(out=0), dict(sg=4), dict(su=7), dict(so=7), dict(sg=-16),
             dict(out=P + 16, so=16), dict(out=P + 8, so=16), dict(out=P, so=8)]
    for kw in cases:
        want = geglu(**kw)
        assert want not in (_capi.OK, _capi.ERR_DEVICE), kw
        assert geglu_noalloc(**kw) == want, kw
    assert geglu_noalloc(T=0, gate=0, up=0, out=0) == _capi.OK
    assert geglu_noalloc(F=0) == _capi.OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="host without a GPU only")
@no_device
def test_noalloc_gelu_and_mul_valid_call_reaches_device_check(lib):
    assert geglu_noalloc() == _capi.ERR_DEVICE
    assert geglu_noalloc(out=P, so=16) == _capi.ERR_DEVICE   # in place
