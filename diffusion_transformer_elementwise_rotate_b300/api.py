"""torch-tensor front end of the C ABI (argument marshalling only).

Every function takes CUDA tensors on the current device, passes their data
pointers, sizes and element strides to the matching `dtrot_*` entry point, and
enqueues the kernel on torch's current stream of that device.  All arithmetic
runs in libdtrot's sm_103a kernels.

  rope_cos_sin_precompute(freqs)         -> (cos, sin)   ERNIE-Image page, section 1
  rope_rotate_half(x, cos, sin, out=None) -> out         ERNIE-Image page, section 2
  rope_rotate_half_qk_(q, k, cos=None, sin=None, freqs=None)   q and k in place, one launch;
                                         tables, or angles evaluated in the kernel
  gelu_and_mul(gate, up, out=None, workspace=None, table=None) -> out   ERNIE-Image page, section 3
  gelu_table(device)                      -> the activation table, built once per device
  gelu_table_build(table)                 -> fills a caller buffer with the activation table
  gelu_and_mul_fused(gate_up, out=None)   -> out         (gate = first half of the last dim)
  gemm_gelu_and_mul(x, w, out=None, workspace=None, check=False) -> out   GEGLU in the
                                         epilogue of the gate_up projection x w^T (tcgen05
                                         tensor cores); check=True reads the kernel's
                                         error word and raises on a failure
  gemm_error_word(workspace)              -> the error word of the last call on it
  rmsnorm_residual(x, residual, w, eps=1e-6, out=None) -> out   (residual updated in place)
                                                         sequence-parallelism post
"""
from __future__ import annotations

import threading

import torch

from . import _capi
from . import selfcheck as _sc

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _last_contiguous(t: torch.Tensor, name: str) -> None:
    if t.dim() and t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")


def rope_cos_sin_precompute(freqs: torch.Tensor, cos_out: torch.Tensor | None = None,
                            sin_out: torch.Tensor | None = None):
    """freqs fp32 (S, B, 1, R) -> cos, sin bf16 (B*S, R)."""
    _need(freqs, "freqs", torch.float32)
    if freqs.dim() != 4 or freqs.shape[2] != 1:
        raise ValueError("freqs must be (S, B, 1, R)")
    if not freqs.is_contiguous():
        raise ValueError("freqs must be contiguous")
    S, B, _, R = freqs.shape
    if cos_out is None:
        cos_out = torch.empty((B * S, R), dtype=torch.bfloat16, device=freqs.device)
    if sin_out is None:
        sin_out = torch.empty((B * S, R), dtype=torch.bfloat16, device=freqs.device)
    for t, n in ((cos_out, "cos_out"), (sin_out, "sin_out")):
        _need(t, n, torch.bfloat16)
        if t.shape != (B * S, R) or not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous (B*S, R)")
    _capi.check("dtrot_rope_cos_sin_precompute", freqs.data_ptr(), S, B, R, cos_out.data_ptr(),
                sin_out.data_ptr(), _stream(freqs))
    if _sc.want("rope_cos_sin_precompute", freqs):
        rc, rs = _sc.ref_tables(freqs)
        _sc.compare("rope_cos_sin_precompute cos", cos_out, rc, exact=False)
        _sc.compare("rope_cos_sin_precompute sin", sin_out, rs, exact=False)
    return cos_out, sin_out


def rope_rotate_half(x: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """x bf16 (B, S, H, D) (any strides, D contiguous); cos/sin bf16 (B*S, rot)."""
    _need(x, "x", torch.bfloat16)
    _need(cos, "cos", torch.bfloat16)
    _need(sin, "sin", torch.bfloat16)
    if x.dim() != 4:
        raise ValueError("x must be (B, S, H, D)")
    _last_contiguous(x, "x")
    B, S, H, D = x.shape
    if cos.dim() != 2 or cos.shape != sin.shape or cos.shape[0] != B * S:
        raise ValueError("cos/sin must be (B*S, rot_dim)")
    if not (cos.is_contiguous() and sin.is_contiguous()):
        raise ValueError("cos/sin must be contiguous")
    rot = cos.shape[1]
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16)
    if out.shape != x.shape:
        raise ValueError("out must have the shape of x")
    _last_contiguous(out, "out")
    sx, so = x.stride(), out.stride()
    key = _sc.want("rope_rotate_half", x, cos)
    x0 = x.clone() if key else None
    _capi.check("dtrot_rope_rotate_half", x.data_ptr(), B, S, H, D, sx[0], sx[1], sx[2],
                cos.data_ptr(), sin.data_ptr(), rot, out.data_ptr(), so[0], so[1], so[2],
                _stream(x))
    if key:
        _sc.compare("rope_rotate_half", out, _sc.ref_rope(x0, cos, sin), exact=True)
    return out


def _qk_args(q, k, cos, sin, freqs):
    """Shapes of a q+k RoPE call and the pointers of its tables or angles:
    (B, S, Hq, Hk, D, rot, cos_ptr, sin_ptr, freqs_ptr), 0 for a pointer not
    given."""
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be (B, S, H, D)")
    if q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q and k must share B, S and D")
    _last_contiguous(q, "q")
    _last_contiguous(k, "k")
    B, S, Hq, D = q.shape
    Hk = k.shape[2]
    if (freqs is None) == (cos is None and sin is None):
        raise ValueError("give either cos and sin, or freqs")
    if freqs is not None:
        _need(freqs, "freqs", torch.float32)
        if freqs.dim() != 4 or freqs.shape[:3] != (S, B, 1) or not freqs.is_contiguous():
            raise ValueError("freqs must be contiguous (S, B, 1, rot)")
        return B, S, Hq, Hk, D, freqs.shape[3], 0, 0, freqs.data_ptr()
    _need(cos, "cos", torch.bfloat16)
    _need(sin, "sin", torch.bfloat16)
    if cos.dim() != 2 or cos.shape != sin.shape or cos.shape[0] != B * S:
        raise ValueError("cos/sin must be (B*S, rot_dim)")
    if not (cos.is_contiguous() and sin.is_contiguous()):
        raise ValueError("cos/sin must be contiguous")
    return B, S, Hq, Hk, D, cos.shape[1], cos.data_ptr(), sin.data_ptr(), 0


def _qk_selfcheck(pairs, cos, sin, freqs):
    """First-call check of a q+k RoPE call: each (name, input copy, output)
    against the plain torch reference."""
    if freqs is not None:
        cos, sin = _sc.ref_tables(freqs)
    for name, x0, out in pairs:
        _sc.compare(name, out, _sc.ref_rope(x0, cos, sin), exact=True)


def rope_rotate_half_qk_(q: torch.Tensor, k: torch.Tensor, cos: torch.Tensor | None = None,
                         sin: torch.Tensor | None = None,
                         freqs: torch.Tensor | None = None) -> None:
    """Rotates q (B, S, Hq, D) and k (B, S, Hk, D) in place with one launch.
    Give either the cos/sin tables (bf16 (B*S, rot)) or the angles `freqs`
    (fp32 (S, B, 1, rot)), from which the kernel evaluates the rows itself.
    q and k may be the q and k head ranges of one fused QKV tensor."""
    B, S, Hq, Hk, D, rot, cp, sp, fp = _qk_args(q, k, cos, sin, freqs)
    sq, sk = q.stride(), k.stride()
    key = _sc.want("rope_rotate_half_qk", q, k, cos if freqs is None else freqs)
    q0, k0 = (q.clone(), k.clone()) if key else (None, None)
    _capi.check("dtrot_rope_rotate_half_qk", q.data_ptr(), Hq, sq[0], sq[1], sq[2],
                k.data_ptr(), Hk, sk[0], sk[1], sk[2], B, S, D, cp or None, sp or None,
                fp or None, rot, _stream(q))
    if key:
        _qk_selfcheck([("rope_rotate_half_qk q", q0, q), ("rope_rotate_half_qk k", k0, k)],
                      cos, sin, freqs)


def rope_rotate_half_qk(q: torch.Tensor, k: torch.Tensor, cos: torch.Tensor | None = None,
                        sin: torch.Tensor | None = None, freqs: torch.Tensor | None = None,
                        q_out: torch.Tensor | None = None,
                        k_out: torch.Tensor | None = None):
    """Rotates q (B, S, Hq, D) into q_out and k (B, S, Hk, D) into k_out with
    one launch, tail columns copied: each output equals rope_rotate_half of its
    input.  Tables or angles as for rope_rotate_half_qk_.  The outputs are
    allocated when not given (any strides with D contiguous otherwise).
    Returns (q_out, k_out)."""
    B, S, Hq, Hk, D, rot, cp, sp, fp = _qk_args(q, k, cos, sin, freqs)
    if q_out is None:
        q_out = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=q.device)
    if k_out is None:
        k_out = torch.empty((B, S, Hk, D), dtype=torch.bfloat16, device=k.device)
    for t, name, like in ((q_out, "q_out", q), (k_out, "k_out", k)):
        _need(t, name, torch.bfloat16)
        if t.shape != like.shape:
            raise ValueError(f"{name} must have the shape of {name[0]}")
        _last_contiguous(t, name)
    sq, sk, soq, sok = q.stride(), k.stride(), q_out.stride(), k_out.stride()
    key = _sc.want("rope_rotate_half_qk_out", q, k, cos if freqs is None else freqs)
    _capi.check("dtrot_rope_rotate_half_qk_out", q.data_ptr(), Hq, sq[0], sq[1], sq[2],
                k.data_ptr(), Hk, sk[0], sk[1], sk[2], B, S, D, cp or None, sp or None,
                fp or None, rot, q_out.data_ptr(), soq[0], soq[1], soq[2], k_out.data_ptr(),
                sok[0], sok[1], sok[2], _stream(q))
    if key:
        _qk_selfcheck([("rope_rotate_half_qk q", q, q_out),
                            ("rope_rotate_half_qk k", k, k_out)], cos, sin, freqs)
    return q_out, k_out


def _rows(t: torch.Tensor, name: str):
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D (rows, features)")
    _last_contiguous(t, name)
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def gelu_workspace(device: torch.device, stream: int) -> torch.Tensor:
    """The GEGLU workspace used for calls on (device, stream): one buffer per
    stream, so calls that may overlap on the GPU never share one."""
    key = (torch.device(device).index, int(stream))
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None:
            n = int(_capi.load().dtrot_gelu_and_mul_workspace_bytes())
            ws = torch.empty(n, dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
    return ws


_tables: dict = {}


def gelu_table_build(table: torch.Tensor) -> torch.Tensor:
    """Fill `table` (a CUDA buffer of at least dtrot_gelu_and_mul_workspace_bytes()
    bytes, 16-byte aligned) with the GEGLU activation table on the current
    stream; gelu_and_mul(..., table=table) then runs the streaming kernel
    alone.  gelu_and_mul(gate, up, workspace=ws) is this followed by
    gelu_and_mul(gate, up, table=ws)."""
    if not isinstance(table, torch.Tensor) or not table.is_cuda:
        raise ValueError("table must be a CUDA tensor")
    _capi.check("dtrot_gelu_table_build", table.data_ptr(),
                table.numel() * table.element_size(), _stream(table))
    return table


def gelu_table(device) -> torch.Tensor:
    """The activation table of `device`, built once (on the current stream,
    with an event that later calls on other streams wait for) and kept."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    with _ws_lock:
        entry = _tables.get(idx)
        if entry is None:
            n = int(_capi.load().dtrot_gelu_and_mul_workspace_bytes())
            dev = torch.device("cuda", idx)
            tab = torch.empty(n, dtype=torch.uint8, device=dev)
            st = torch.cuda.current_stream(dev)
            _capi.check("dtrot_gelu_table_build", tab.data_ptr(), n, st.cuda_stream)
            ready = torch.cuda.Event()
            ready.record(st)
            entry = (tab, ready)
            _tables[idx] = entry
    tab, ready = entry
    torch.cuda.current_stream(tab.device).wait_event(ready)
    return tab


def gelu_and_mul(gate: torch.Tensor, up: torch.Tensor, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None,
                 table: torch.Tensor | None = None) -> torch.Tensor:
    """gate, up bf16 (T, F) (row strides allowed) -> out bf16 (T, F).
    `workspace` (a CUDA buffer of dtrot_gelu_and_mul_workspace_bytes() bytes)
    defaults to a buffer cached per device and stream; the call builds the
    activation table there.  With `table` (from gelu_table()), the table is
    not rebuilt."""
    _need(gate, "gate", torch.bfloat16)
    _need(up, "up", torch.bfloat16)
    if gate.shape != up.shape:
        raise ValueError("gate and up must have the same shape")
    T, F = gate.shape
    sg, su = _rows(gate, "gate"), _rows(up, "up")
    if out is None:
        out = torch.empty((T, F), dtype=torch.bfloat16, device=gate.device)
    _need(out, "out", torch.bfloat16)
    if out.shape != gate.shape:
        raise ValueError("out must be (T, F)")
    so = _rows(out, "out")
    st = _stream(gate)
    if table is not None:
        if not table.is_cuda:
            raise ValueError("table must be a CUDA tensor")
        key = _sc.want("gelu_and_mul", gate, up)
        ref = _sc.ref_geglu(gate, up) if key else None
        _capi.check("dtrot_gelu_and_mul_with_table", gate.data_ptr(), sg, up.data_ptr(), su,
                    out.data_ptr(), so, T, F, table.data_ptr(),
                    table.numel() * table.element_size(), st)
        if key:
            _sc.compare("gelu_and_mul", out, ref, exact=False)
        return out
    if workspace is None:
        workspace = gelu_workspace(gate.device, st)
    elif not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    key = _sc.want("gelu_and_mul", gate, up)
    ref = _sc.ref_geglu(gate, up) if key else None
    _capi.check("dtrot_gelu_and_mul", gate.data_ptr(), sg, up.data_ptr(), su, out.data_ptr(),
                so, T, F, workspace.data_ptr(), nbytes, st)
    if key:
        _sc.compare("gelu_and_mul", out, ref, exact=False)
    return out


def _cached_workspace(kind: str, query: str, device: torch.device, stream: int) -> torch.Tensor:
    key = (kind, torch.device(device).index, int(stream))
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None:
            n = int(getattr(_capi.load(), query)())
            ws = torch.empty(n, dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
    return ws


def gemm_error_word(workspace: torch.Tensor) -> int:
    """The error word a gemm_gelu_and_mul call left in `workspace` (0: every
    wait completed and the output is valid; see dtrot_gemm_gelu_and_mul_error).
    Reads it on the current stream, after the calls queued there, and waits
    for that read."""
    import ctypes
    word = ctypes.c_uint32(0)
    st = torch.cuda.current_stream(workspace.device)
    _capi.check("dtrot_gemm_gelu_and_mul_error", workspace.data_ptr(), ctypes.addressof(word),
                st.cuda_stream)
    st.synchronize()
    return int(word.value)


def gemm_gelu_and_mul(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None,
                      gate_up: torch.Tensor | None = None, check: bool = False,
                      _withhold_last_stage: bool = False) -> torch.Tensor:
    """GEGLU of the MLP's gate_up projection without storing gate_up:
    x bf16 (T, C), w bf16 (2F, C) (gate rows first) -> out bf16 (T, F) =
    up * gelu(gate) with gate_up = x w^T rounded to bf16.  If `gate_up` (bf16
    (T, 2F)) is given, the rounded projection is stored there as well.
    With check=True the call waits for the kernel and raises DtrotKernelError
    if it reported a failure in its error word (a wait that ran out of time);
    `_withhold_last_stage` runs the diagnostic variant whose last pipeline
    stage is never loaded (tests only)."""
    _need(x, "x", torch.bfloat16)
    _need(w, "w", torch.bfloat16)
    if x.dim() != 2 or w.dim() != 2 or w.shape[1] != x.shape[1] or w.shape[0] % 2:
        raise ValueError("x must be (T, C) and w (2F, C)")
    if not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("x and w must be contiguous")
    T, C = x.shape
    F = w.shape[0] // 2
    if out is None:
        out = torch.empty((T, F), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16)
    if out.shape != (T, F):
        raise ValueError("out must be (T, F)")
    so = _rows(out, "out")
    st = _stream(x)
    if workspace is None:
        workspace = _cached_workspace("gemm_geglu", "dtrot_gemm_gelu_and_mul_workspace_bytes",
                                      x.device, st)
    gp, sgu = 0, 2 * F
    if gate_up is not None:
        _need(gate_up, "gate_up", torch.bfloat16)
        if gate_up.shape != (T, 2 * F):
            raise ValueError("gate_up must be (T, 2F)")
        gp, sgu = gate_up.data_ptr(), _rows(gate_up, "gate_up")
    key = _sc.want("gemm_gelu_and_mul", x, w)
    entry = ("dtrot_gemm_gelu_and_mul_withhold_last_stage" if _withhold_last_stage
             else "dtrot_gemm_gelu_and_mul")
    _capi.check(entry, x.data_ptr(), T, C, w.data_ptr(), F, out.data_ptr(),
                so, gp or None, sgu, workspace.data_ptr(),
                workspace.numel() * workspace.element_size(), st)
    if check:
        word = gemm_error_word(workspace)
        if word:
            raise _capi.DtrotKernelError(
                f"gemm_gelu_and_mul: the kernel reported error word {word:#x} "
                "(1: free stage, 2: loaded stage, 4: accumulator wait ran out of time; "
                "8: CTA pair tensor-memory mismatch); its output is not valid")
    if key:
        def rerun(rows):
            o = torch.empty((rows, F), dtype=torch.bfloat16, device=x.device)
            g = torch.empty((rows, 2 * F), dtype=torch.bfloat16, device=x.device)
            _capi.check("dtrot_gemm_gelu_and_mul", x.data_ptr(), rows, C, w.data_ptr(), F,
                        o.data_ptr(), F, g.data_ptr(), 2 * F, workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), st)
            return o, g

        _sc.check_gemm_geglu(x, w, out, rerun)
    return out


def gelu_and_mul_fused(gate_up: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """(..., 2F) buffer, gate = [..., :F], up = [..., F:] -> (..., F)."""
    if gate_up.shape[-1] % 2:
        raise ValueError("the last dimension of gate_up must be even")
    F = gate_up.shape[-1] // 2
    g2 = gate_up.reshape(-1, 2 * F)
    o2 = None if out is None else out.view(-1, F)
    r = gelu_and_mul(g2[:, :F], g2[:, F:], o2)
    return r.view(*gate_up.shape[:-1], F)


def rmsnorm_residual(x: torch.Tensor, residual: torch.Tensor, w: torch.Tensor,
                     eps: float = 1e-6, out: torch.Tensor | None = None) -> torch.Tensor:
    """x, residual bf16 (T, C); w bf16 (C,).  residual is overwritten with
    h = x + residual; returns out = RMSNorm(h) * w."""
    _need(x, "x", torch.bfloat16)
    _need(residual, "residual", torch.bfloat16)
    _need(w, "w", torch.bfloat16)
    if x.shape != residual.shape or w.dim() != 1 or w.shape[0] != x.shape[-1]:
        raise ValueError("shapes: x (T, C), residual (T, C), w (C,)")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    T, C = x.shape
    sx, sr = _rows(x, "x"), _rows(residual, "residual")
    if out is None:
        out = torch.empty((T, C), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16)
    so = _rows(out, "out")
    key = _sc.want("rmsnorm_residual", x, w)
    ref = _sc.ref_rmsnorm(x, residual, w, eps) if key else None
    _capi.check("dtrot_rmsnorm_residual", x.data_ptr(), sx, residual.data_ptr(), sr,
                w.data_ptr(), float(eps), out.data_ptr(), so, T, C, _stream(x))
    if key:
        _sc.compare("rmsnorm_residual residual", residual, ref[0], exact=True)
        _sc.compare("rmsnorm_residual out", out, ref[1], exact=False)
    return out
