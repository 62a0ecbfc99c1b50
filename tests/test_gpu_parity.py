"""GPU kernels (through the C ABI) against the CPU oracle, element by element.

Bars: RoPE and the cos/sin tables bit-exact; GEGLU and RMSNorm within 1 bf16
ulp everywhere with at most 0.01% of elements different (both are expected to
be bit-exact by design; the mismatch count is printed).  Inputs are the seeded
synthetic workloads; the full-size video layer runs in the launch
configuration the benchmark times and is checked on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import diffusion_transformer_elementwise_rotate_b300 as dt
from diffusion_transformer_elementwise_rotate_b300 import workloads as W
from _compare import assert_bitexact, assert_within_tolerance, ulp_diff

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = float(np.float32(1e-6))
bits = oracle.bf16_bits


def to_dev(t):
    return t.to(DEV, non_blocking=False)


def from_u16(a):
    return oracle.from_bits(a)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dt.load()
    torch.cuda.init()


# ---------------------------------------------------------------- cos/sin tables

@pytest.mark.parametrize("name", ["tiny", "image", "cfg", "video"])
def test_cos_sin_tables_bitexact(name):
    wl = W.WORKLOADS[name]
    freqs = W.freqs_for(wl)
    c, s = dt.rope_cos_sin_precompute(to_dev(freqs))
    ec, es = oracle.rope_cos_sin(freqs.numpy())
    assert_bitexact(bits(c), ec, f"{name} cos")
    assert_bitexact(bits(s), es, f"{name} sin")


@pytest.mark.parametrize("shape", [(3, 5, 1, 6), (7, 2, 1, 16), (1000, 1, 1, 8)])
def test_cos_sin_random_and_special_angles(shape):
    g = torch.Generator().manual_seed(17)
    n = int(np.prod(shape))
    f = torch.empty(n, dtype=torch.float32)
    f.uniform_(-200.0, 200.0, generator=g)
    special = torch.tensor([0.0, -0.0, 1e-30, -1e-40, 1.5707964, 3.1415927, 4.712389, 1e4,
                            -3.3e4, 1e6, 1e30, float("inf"), float("-inf"), float("nan")])
    k = min(n, special.numel())
    f[:k] = special[:k]
    f = f.view(*shape)
    c, s = dt.rope_cos_sin_precompute(to_dev(f))
    ec, es = oracle.rope_cos_sin(f.numpy())
    assert_bitexact(bits(c), ec, "cos")
    assert_bitexact(bits(s), es, "sin")


def test_cos_sin_many_angles_near_rounding_midpoints():
    # 4M angles spread over the position * frequency range of the workloads
    g = torch.Generator().manual_seed(5)
    f = (torch.rand(1 << 22, generator=g) * 60.0 - 5.0).view(-1, 1, 1, 64)
    c, s = dt.rope_cos_sin_precompute(to_dev(f))
    ec, es = oracle.rope_cos_sin(f.numpy())
    assert_bitexact(bits(c), ec, "cos")
    assert_bitexact(bits(s), es, "sin")


def test_cos_sin_second_half_reused_only_for_identical_bits():
    # rows of 32 angles (R % 16 == 0: the kernel pairs column j with j + 16 and
    # copies j's entry when the two angles have the same bits): equal halves,
    # halves that differ in one column, +0 against -0 (equal values, different
    # sin), NaNs with different payloads, and random halves
    g = torch.Generator().manual_seed(29)
    S, B, R = 515, 2, 32
    f = (torch.rand((S, B, 1, R), generator=g) * 400.0 - 200.0)
    f[: S // 2, :, :, R // 2:] = f[: S // 2, :, :, : R // 2]
    f[1::7, :, :, R // 2 + 3] += 1.0
    f[2, 0, 0, 5], f[2, 0, 0, R // 2 + 5] = 0.0, -0.0
    f[3, 1, 0, 6], f[3, 1, 0, R // 2 + 6] = -0.0, 0.0
    nan_a = np.array([0x7FC00001], dtype=np.uint32).view(np.float32)[0]
    nan_b = np.array([0xFFC00002], dtype=np.uint32).view(np.float32)[0]
    f[4, 0, 0, 1], f[4, 0, 0, R // 2 + 1] = float(nan_a), float(nan_b)
    f = f.contiguous()
    c, s = dt.rope_cos_sin_precompute(to_dev(f))
    ec, es = oracle.rope_cos_sin(f.numpy())
    assert_bitexact(bits(c), ec, "cos")
    assert_bitexact(bits(s), es, "sin")


def test_cos_sin_reduction_range_and_zero_crossings():
    # Angles where the table kernel's hardware sine/cosine path ends: uniform over
    # [-4100, 4100] (that path reduces |f| <= 4096 by 2 pi), next to every multiple
    # of pi/2 up to 4096 (zeros of sin and cos, and the ends of the reduced
    # range), and the float32 neighbours of +-4096.
    g = torch.Generator().manual_seed(23)
    u = torch.rand(1 << 21, generator=g, dtype=torch.float64) * 8200.0 - 4100.0
    base = torch.arange(-2608, 2609, dtype=torch.float64) * (math.pi / 2)
    near = torch.cat([base + d for d in (-1e-3, -3e-5, -1e-6, 0.0, 1e-6, 3e-5, 1e-3)])
    e = np.array([4096.0, -4096.0], dtype=np.float32)
    edge = np.concatenate([e, np.nextafter(e, np.float32(0)), np.nextafter(e, e * 2)])
    f = torch.cat([u.to(torch.float32), near.to(torch.float32), torch.from_numpy(edge)])
    f = f[: (f.numel() // 8) * 8].reshape(-1, 1, 1, 8).contiguous()
    c, s = dt.rope_cos_sin_precompute(to_dev(f))
    ec, es = oracle.rope_cos_sin(f.numpy())
    assert_bitexact(bits(c), ec, "cos")
    assert_bitexact(bits(s), es, "sin")


# ---------------------------------------------------------------- RoPE

def _rope_case(x, cos_b, sin_b, **kw):
    got = dt.rope_rotate_half(to_dev(x), to_dev(from_u16(cos_b)), to_dev(from_u16(sin_b)), **kw)
    return bits(got)


@pytest.mark.parametrize("name", ["tiny", "image", "cfg"])
@pytest.mark.parametrize("which", ["q", "k"])
def test_rope_configs_bitexact(name, which):
    wl = W.WORKLOADS[name]
    x = W.rope_inputs(wl, which)
    cos_b, sin_b = oracle.rope_cos_sin(W.freqs_for(wl).numpy())
    exp = oracle.rope_rotate_half(bits(x), cos_b, sin_b)
    assert_bitexact(_rope_case(x, cos_b, sin_b), exp, f"{name} {which}")


def test_rope_video_full_size_sampled_tokens():
    wl = W.WORKLOADS["video"]
    x = W.rope_inputs(wl, "q")
    freqs = W.freqs_for(wl)
    cd, sd = dt.rope_cos_sin_precompute(to_dev(freqs))
    out = dt.rope_rotate_half(to_dev(x), cd, sd)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(wl.S, 1024, replace=False))
    toks = np.concatenate([[0, wl.S - 1], toks])
    cos_b, sin_b = bits(cd)[toks], bits(sd)[toks]
    xs = bits(x)[:, toks]
    exp = oracle.rope_rotate_half(xs, cos_b, sin_b)
    assert_bitexact(bits(out)[:, toks], exp, "video sampled")


SWEEP = [(64, 32), (64, 48), (64, 64), (80, 40), (80, 60), (80, 80), (128, 64), (128, 96),
         (128, 128)]


@pytest.mark.parametrize("D,rot", SWEEP)
def test_rope_sweep_odd_S(D, rot):
    B, S = 1, 4097
    H = max(1, (1 << 20) // (S * D))
    x = W.normal_bf16((B, S, H, D), 40 + D + rot, 0)
    cos_b, sin_b = oracle.rope_cos_sin(W.freqs_1d(S, B, rot).numpy())
    exp = oracle.rope_rotate_half(bits(x), cos_b, sin_b)
    assert_bitexact(_rope_case(x, cos_b, sin_b), exp, f"D={D} rot={rot}")


def test_rope_unrelated_table_halves_strided_qkv_and_misaligned():
    rng = np.random.default_rng(3)
    B, S, H, D, rot = 2, 37, 3, 128, 96
    qkv = W.normal_bf16((B, S, 3 * H, D), 21, 0)
    cos_b = oracle.rn16_array(rng.uniform(-2, 2, (B * S, rot)))
    sin_b = oracle.rn16_array(rng.uniform(-2, 2, (B * S, rot)))
    dq = to_dev(qkv)
    k_view = dq[:, :, H:2 * H]                      # strided view, 16-byte aligned
    got = dt.rope_rotate_half(k_view, to_dev(from_u16(cos_b)), to_dev(from_u16(sin_b)))
    exp = oracle.rope_rotate_half(bits(qkv)[:, :, H:2 * H], cos_b, sin_b)
    assert_bitexact(bits(got), exp, "strided k")
    # one element off the 16-byte grid: the scalar path
    flat = torch.empty(B * S * H * D + 1, dtype=torch.bfloat16, device=DEV)
    xm = flat[1:].view(B, S, H, D)
    xm.copy_(dq[:, :, :H])
    om = torch.empty(B * S * H * D + 1, dtype=torch.bfloat16, device=DEV)[1:].view(B, S, H, D)
    dt.rope_rotate_half(xm, to_dev(from_u16(cos_b)), to_dev(from_u16(sin_b)), out=om)
    exp = oracle.rope_rotate_half(bits(qkv)[:, :, :H], cos_b, sin_b)
    assert_bitexact(bits(om), exp, "misaligned")


@pytest.mark.parametrize("D,rot", [(128, 96), (80, 60), (64, 64)])
def test_rope_in_place(D, rot):
    B, S, H = 1, 333, 5
    x = W.normal_bf16((B, S, H, D), 7, 1)
    cos_b, sin_b = oracle.rope_cos_sin(W.freqs_1d(S, B, rot).numpy())
    xd = to_dev(x)
    r = dt.rope_rotate_half(xd, to_dev(from_u16(cos_b)), to_dev(from_u16(sin_b)), out=xd)
    assert r.data_ptr() == xd.data_ptr()
    assert_bitexact(bits(xd), oracle.rope_rotate_half(bits(x), cos_b, sin_b), "in place")


def test_rope_exhaustive_x_and_special_values():
    allx = np.arange(1 << 16, dtype=np.uint16)
    partner = np.roll(allx, 12345)
    x = np.stack([allx, partner], axis=-1).reshape(1, -1, 1, 2)
    S = x.shape[1]
    cases = [(0x3F80, 0x0000), (0x3F35, 0x3F35), (0xBE9A, 0x3F74), (0x3C23, 0xBF7F),
             (0x0001, 0x0081), (0x7F80, 0x3F00), (0x7FC0, 0x0000), (0x1F80, 0x2000)]
    for c, s in cases:
        cos_b = np.full((S, 2), c, np.uint16)
        sin_b = np.full((S, 2), s, np.uint16)
        got = _rope_case(from_u16(x), cos_b, sin_b)
        assert_bitexact(got, oracle.rope_rotate_half(x, cos_b, sin_b), f"c={c:#x} s={s:#x}")


def test_rope_empty():
    x = torch.empty((1, 0, 4, 64), dtype=torch.bfloat16, device=DEV)
    c = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    out = dt.rope_rotate_half(x, c, c)
    assert out.shape == x.shape


# ---------------------------------------------------------------- q and k in one launch

def _qk_check(B, S, Hq, Hk, D, rot, freqs, seed, mode, layout="qkv", offset=0, out=None):
    """RoPE on q and k in one launch against the oracle on each: in place
    (out=None), or out of place into separate outputs with padded head rows
    (out="separate") or into the q and k head ranges of one output buffer
    (out="fused"); out of place, the inputs and the padding stay unchanged."""
    Hv = Hq if layout == "qkv" else 0
    if layout == "qkv":
        buf = W.normal_bf16((B, S, Hq + Hk + Hv, D), seed, 0)
        dbuf = to_dev(buf)
        if offset:
            flat = torch.empty(dbuf.numel() + offset, dtype=torch.bfloat16, device=DEV)
            view = flat[offset:].view(dbuf.shape)
            view.copy_(dbuf)
            dbuf = view
        q, k, v = dbuf[:, :, :Hq], dbuf[:, :, Hq:Hq + Hk], dbuf[:, :, Hq + Hk:]
        q0, k0 = bits(buf)[:, :, :Hq], bits(buf)[:, :, Hq:Hq + Hk]
        v0 = bits(buf)[:, :, Hq + Hk:]
    else:
        qh = W.normal_bf16((B, S, Hq, D), seed, 0)
        kh = W.normal_bf16((B, S, Hk, D), seed, 1)
        q, k, v = to_dev(qh), to_dev(kh), None
        q0, k0 = bits(qh), bits(kh)
    ec, es = oracle.rope_cos_sin(freqs.numpy())
    if mode == "angles":
        kw = {"freqs": to_dev(freqs)}
    else:
        kw = {"cos": to_dev(from_u16(ec)), "sin": to_dev(from_u16(es))}
    if out is None:
        dt.rope_rotate_half_qk_(q, k, **kw)
        rq, rk = q, k
    else:
        pad = 0 if out == "fused" else 16
        nan = float("nan")
        if out == "fused":
            obuf = torch.full((B, S, Hq + Hk, D), nan, dtype=torch.bfloat16, device=DEV)
            qo, ko = obuf[:, :, :Hq], obuf[:, :, Hq:]
        else:
            qpad = torch.full((B, S, Hq, D + pad), nan, dtype=torch.bfloat16, device=DEV)
            kpad = torch.full((B, S, Hk, D + pad), nan, dtype=torch.bfloat16, device=DEV)
            qo, ko = qpad[..., :D], kpad[..., :D]
        rq, rk = dt.rope_rotate_half_qk(q, k, q_out=qo, k_out=ko, **kw)
        assert rq is qo and rk is ko
        torch.cuda.synchronize()
        assert_bitexact(bits(q), q0, "q input unchanged")
        assert_bitexact(bits(k), k0, "k input unchanged")
        if pad:
            for t in (qpad, kpad):
                assert (bits(t)[..., D:] == 0x7FC0).all(), "padding written"
    torch.cuda.synchronize()
    assert_bitexact(bits(rq), oracle.rope_rotate_half(q0, ec, es), f"q {mode} {out}")
    assert_bitexact(bits(rk), oracle.rope_rotate_half(k0, ec, es), f"k {mode} {out}")
    if v is not None:
        assert_bitexact(bits(v), v0, "v untouched")


@pytest.mark.parametrize("mode", ["tables", "angles"])
@pytest.mark.parametrize("name", ["tiny", "image", "cfg"])
def test_rope_qk_fused_qkv_configs(name, mode):
    wl = W.WORKLOADS[name]
    _qk_check(wl.B, wl.S, wl.H, wl.H, wl.D, wl.rot, W.freqs_for(wl), wl.seed + 50, mode)


@pytest.mark.parametrize("mode", ["tables", "angles"])
@pytest.mark.parametrize("D,rot", SWEEP)
def test_rope_qk_sweep_odd_S_gqa(D, rot, mode):
    B, S = 1, 4097
    _qk_check(B, S, 6, 2, D, rot, W.freqs_1d(S, B, rot), 90 + D + rot, mode)


@pytest.mark.parametrize("mode", ["tables", "angles"])
def test_rope_qk_separate_buffers_misaligned_and_wide(mode):
    _qk_check(2, 37, 3, 5, 128, 96, W.freqs_1d(37, 2, 96), 7, mode, layout="separate")
    _qk_check(2, 37, 3, 3, 128, 96, W.freqs_1d(37, 2, 96), 8, mode, offset=1)  # scalar path
    _qk_check(1, 19, 2, 2, 640, 576, W.freqs_1d(19, 1, 576), 9, mode)          # rot > 256


def test_rope_qk_special_angles_match_the_table_kernel():
    g = torch.Generator().manual_seed(23)
    f = torch.empty(64 * 32, dtype=torch.float32).uniform_(-300.0, 300.0, generator=g)
    special = torch.tensor([0.0, -0.0, 1e-30, 1.5707964, 3.1415927, 1e4, -3.3e4, 1e6, 1e30,
                            float("inf"), float("-inf"), float("nan")])
    f[:special.numel()] = special
    freqs = f.view(64, 1, 1, 32)
    _qk_check(1, 64, 2, 2, 32, 32, freqs, 10, "angles")


def test_rope_qk_angles_second_half_reused_only_for_identical_bits():
    # angle mode evaluates column j of the first half and copies the entry to
    # j + rot/2 when that angle has the same bits: equal halves, one column off,
    # +0 against -0, NaN payloads, and random halves, checked against the
    # oracle's tables
    g = torch.Generator().manual_seed(31)
    S, B, R = 131, 2, 64
    f = torch.rand((S, B, 1, R), generator=g) * 400.0 - 200.0
    f[: S // 2, :, :, R // 2:] = f[: S // 2, :, :, : R // 2]
    f[1::5, :, :, R // 2 + 3] += 1.0
    f[2, 0, 0, 5], f[2, 0, 0, R // 2 + 5] = 0.0, -0.0
    f[3, 1, 0, 6], f[3, 1, 0, R // 2 + 6] = -0.0, 0.0
    nan_a = np.array([0x7FC00001], dtype=np.uint32).view(np.float32)[0]
    nan_b = np.array([0xFFC00002], dtype=np.uint32).view(np.float32)[0]
    f[4, 0, 0, 1], f[4, 0, 0, R // 2 + 1] = float(nan_a), float(nan_b)
    _qk_check(B, S, 3, 2, R, R, f.contiguous(), 77, "angles")


@pytest.mark.parametrize("out", ["separate", "fused"])
@pytest.mark.parametrize("mode", ["tables", "angles"])
@pytest.mark.parametrize("name", ["tiny", "image", "cfg"])
def test_rope_qk_out_of_place_configs(name, mode, out):
    # image: rot 96 of D 128, so out of place the tail columns are copied
    wl = W.WORKLOADS[name]
    _qk_check(wl.B, wl.S, wl.H, wl.H, wl.D, wl.rot, W.freqs_for(wl), wl.seed + 60, mode,
              out=out)


@pytest.mark.parametrize("mode", ["tables", "angles"])
@pytest.mark.parametrize("D,rot", SWEEP)
def test_rope_qk_out_of_place_sweep_odd_S_gqa(D, rot, mode):
    B, S = 1, 4097
    _qk_check(B, S, 6, 2, D, rot, W.freqs_1d(S, B, rot), 190 + D + rot, mode, out="separate")


@pytest.mark.parametrize("mode", ["tables", "angles"])
def test_rope_qk_out_of_place_misaligned_wide_and_long_tails(mode):
    _qk_check(2, 37, 3, 5, 128, 96, W.freqs_1d(37, 2, 96), 17, mode, layout="separate",
              out="separate")
    _qk_check(2, 37, 3, 3, 128, 96, W.freqs_1d(37, 2, 96), 18, mode, offset=1,
              out="separate")                                                   # scalar path
    _qk_check(1, 19, 2, 2, 640, 576, W.freqs_1d(19, 1, 576), 19, mode, out="fused")  # rot > 256
    # 4 pair and 56 tail vectors per head row: more items than lanes, generic path
    _qk_check(1, 45, 3, 1, 512, 64, W.freqs_1d(45, 1, 64), 20, mode, out="separate")
    # 4 pair and 4 tail vectors: every lane busy, 4 rows per warp pass
    _qk_check(1, 45, 5, 3, 96, 64, W.freqs_1d(45, 1, 64), 21, mode, out="fused")


def test_rope_qk_out_of_place_equals_rope_rotate_half():
    # the single launch gives what two rope_rotate_half calls give, bit for bit
    wl = W.WORKLOADS["image"]
    freqs = to_dev(W.freqs_for(wl))
    q, k = to_dev(W.rope_inputs(wl, "q")), to_dev(W.rope_inputs(wl, "k"))
    c, s = dt.rope_cos_sin_precompute(freqs)
    qo, ko = dt.rope_rotate_half_qk(q, k, cos=c, sin=s)
    assert np.array_equal(bits(qo), bits(dt.rope_rotate_half(q, c, s)))
    assert np.array_equal(bits(ko), bits(dt.rope_rotate_half(k, c, s)))


@pytest.mark.parametrize("mode", ["angles", "tables"])
def test_rope_qk_out_of_place_video_full_size_sampled_tokens(mode):
    wl = W.WORKLOADS["video"]
    q, k = W.rope_inputs(wl, "q"), W.rope_inputs(wl, "k")
    freqs = W.freqs_for(wl)
    dq, dk = to_dev(q), to_dev(k)
    if mode == "angles":
        qo, ko = dt.rope_rotate_half_qk(dq, dk, freqs=to_dev(freqs))
    else:
        c, s = dt.rope_cos_sin_precompute(to_dev(freqs))
        qo, ko = dt.rope_rotate_half_qk(dq, dk, cos=c, sin=s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    toks = np.unique(np.concatenate([[0, wl.S - 1], rng.choice(wl.S, 512, replace=False)]))
    ec, es = oracle.rope_cos_sin(freqs.numpy()[toks])
    assert_bitexact(bits(qo)[:, toks], oracle.rope_rotate_half(bits(q)[:, toks], ec, es), "q")
    assert_bitexact(bits(ko)[:, toks], oracle.rope_rotate_half(bits(k)[:, toks], ec, es), "k")
    assert_bitexact(bits(dq)[:, toks], bits(q)[:, toks], "q input unchanged")


@pytest.mark.parametrize("mode", ["angles", "tables"])
def test_rope_qk_video_full_size_sampled_tokens(mode):
    wl = W.WORKLOADS["video"]
    q, k = W.rope_inputs(wl, "q"), W.rope_inputs(wl, "k")
    freqs = W.freqs_for(wl)
    dq, dk = to_dev(q), to_dev(k)
    if mode == "angles":
        dt.rope_rotate_half_qk_(dq, dk, freqs=to_dev(freqs))
    else:
        c, s = dt.rope_cos_sin_precompute(to_dev(freqs))
        dt.rope_rotate_half_qk_(dq, dk, cos=c, sin=s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    toks = np.unique(np.concatenate([[0, wl.S - 1], rng.choice(wl.S, 512, replace=False)]))
    ec, es = oracle.rope_cos_sin(freqs.numpy()[toks])
    assert_bitexact(bits(dq)[:, toks], oracle.rope_rotate_half(bits(q)[:, toks], ec, es), "q")
    assert_bitexact(bits(dk)[:, toks], oracle.rope_rotate_half(bits(k)[:, toks], ec, es), "k")


# ---------------------------------------------------------------- GEGLU

def test_geglu_every_bf16_gate_value_bitexact():
    gate = np.arange(1 << 16, dtype=np.uint16).reshape(256, 256)
    up = np.full_like(gate, 0x3F80)
    got = dt.gelu_and_mul(to_dev(from_u16(gate)), to_dev(from_u16(up)))
    assert_bitexact(bits(got), oracle.gelu_and_mul(gate, up), "gelu table")


def test_geglu_every_gate_with_random_up():
    gate = np.arange(1 << 16, dtype=np.uint16).reshape(128, 512)
    up = bits(W.normal_bf16((128, 512), 9, 3, std=3.0))
    up[0, :8] = [0x0001, 0x8001, 0x7F80, 0xFF80, 0x7FC0, 0x0000, 0x8000, 0x7F7F]
    got = bits(dt.gelu_and_mul(to_dev(from_u16(gate)), to_dev(from_u16(up))))
    exp = oracle.gelu_and_mul(gate, up)
    n = assert_within_tolerance(got, exp, "gelu x random up")
    print(f"gelu x random up: {n} mismatches")
    assert_bitexact(got, exp, "gelu x random up (bit-exact by design)")


def _geglu_check(gu, F, rows=None, what=""):
    dgu = to_dev(gu)
    out = dt.gelu_and_mul_fused(dgu)
    torch.cuda.synchronize()
    g = bits(gu)
    if rows is None:
        rows = np.arange(gu.shape[0])
    exp = oracle.gelu_and_mul(g[rows, :F], g[rows, F:])
    got = bits(out)[rows]
    n = assert_within_tolerance(got, exp, what)
    print(f"{what}: {n} mismatches of {got.size}")
    assert_bitexact(got, exp, what)


@pytest.mark.parametrize("name", ["tiny", "image", "cfg", "video"])
def test_geglu_configs(name):
    wl = W.WORKLOADS[name]
    gu = W.geglu_inputs(wl)
    rows = None
    if wl.T_ff > 512:
        rng = np.random.default_rng(1)
        rows = np.unique(np.concatenate([[0, wl.T_ff - 1], rng.choice(wl.T_ff, 384, replace=False)]))
    _geglu_check(gu, wl.F, rows, name)


@pytest.mark.parametrize("F", [768, 2560, 4096, 5120, 12288, 13824, 1001])
def test_geglu_sweep(F):
    T = max(3, (1 << 20) // F) | 1
    gu = W.normal_bf16((T, 2 * F), 60 + F, 2)
    _geglu_check(gu, F, None, f"F={F}")


def test_geglu_separate_buffers_misaligned_and_in_place():
    T, F = 77, 520
    g = W.normal_bf16((T, F + 3), 1, 2)
    u = W.normal_bf16((T, F + 5), 1, 3)
    gd, ud = to_dev(g), to_dev(u)
    # distinct row strides, columns starting one element in (scalar path)
    got = dt.gelu_and_mul(gd[:, 1:F + 1], ud[:, 2:F + 2])
    exp = oracle.gelu_and_mul(bits(g)[:, 1:F + 1], bits(u)[:, 2:F + 2])
    assert_bitexact(bits(got), exp, "misaligned")
    # in place: out == gate
    gate = to_dev(W.normal_bf16((T, F), 2, 2))
    gate0 = bits(gate)
    up = to_dev(W.normal_bf16((T, F), 2, 3))
    r = dt.gelu_and_mul(gate, up, out=gate)
    assert r.data_ptr() == gate.data_ptr()
    assert_bitexact(bits(gate), oracle.gelu_and_mul(gate0, bits(up)), "in place")


def test_geglu_caller_workspace_is_rebuilt_every_call():
    # a caller-owned workspace holding garbage: the call fills in the table itself
    from diffusion_transformer_elementwise_rotate_b300 import _capi
    n = int(_capi.load().dtrot_gelu_and_mul_workspace_bytes())
    gate = np.arange(1 << 16, dtype=np.uint16).reshape(64, 1024)
    up = bits(W.normal_bf16((64, 1024), 11, 3))
    exp = oracle.gelu_and_mul(gate, up)
    for fill in (0xFF, 0x00, 0x7F):
        ws = torch.full((n + 64,), fill, dtype=torch.uint8, device=DEV)[16:16 + n]
        got = dt.gelu_and_mul(to_dev(from_u16(gate)), to_dev(from_u16(up)), workspace=ws)
        assert_bitexact(bits(got), exp, f"workspace filled with {fill:#x}")
    small = torch.empty(n - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(dt.DtrotError):
        dt.gelu_and_mul(to_dev(from_u16(gate)), to_dev(from_u16(up)), workspace=small)


def test_geglu_prebuilt_table_every_gate_value_and_video_rows():
    tab = dt.gelu_table("cuda")
    gate = np.arange(1 << 16, dtype=np.uint16).reshape(128, 512)
    up = bits(W.normal_bf16((128, 512), 13, 3, std=2.0))
    got = dt.gelu_and_mul(to_dev(from_u16(gate)), to_dev(from_u16(up)), table=tab)
    assert_bitexact(bits(got), oracle.gelu_and_mul(gate, up), "prebuilt table, every gate")
    wl = W.WORKLOADS["video"]
    gu = to_dev(W.geglu_inputs(wl))
    F = wl.F
    out = dt.gelu_and_mul(gu[:, :F], gu[:, F:], table=tab)
    ref = dt.gelu_and_mul(gu[:, :F], gu[:, F:])              # the table rebuilt in the call
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    rows = np.unique(np.concatenate([[0, wl.T_ff - 1],
                                     np.random.default_rng(6).choice(wl.T_ff, 64, replace=False)]))
    r = torch.from_numpy(rows).to(DEV)
    g = bits(gu[r])
    assert_bitexact(bits(out[r]), oracle.gelu_and_mul(g[:, :F], g[:, F:]), "prebuilt, video rows")


def test_geglu_empty():
    z = torch.empty((0, 16), dtype=torch.bfloat16, device=DEV)
    assert dt.gelu_and_mul(z, z).shape == (0, 16)


# ---------------------------------------------------------------- RMSNorm

def _rms_check(x, r, w, rows=None, what="", exact=True):
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    y = dt.rmsnorm_residual(xd, rd, wd, EPS)
    torch.cuda.synchronize()
    if rows is None:
        rows = np.arange(x.shape[0])
    h_exp, y_exp = oracle.rmsnorm_residual(bits(x)[rows], bits(r)[rows], bits(w), EPS)
    assert_bitexact(bits(rd)[rows], h_exp, f"{what} residual")
    got = bits(y)[rows]
    n = assert_within_tolerance(got, y_exp, what)
    print(f"{what}: {n} mismatches of {got.size}")
    return n


@pytest.mark.parametrize("name", ["tiny", "image", "cfg", "video"])
@pytest.mark.parametrize("second", [False, True])
def test_rmsnorm_configs(name, second):
    wl = W.WORKLOADS[name]
    x, r, w = W.rmsnorm_inputs(wl, second)
    rows = None
    if wl.T_norm > 512:
        rng = np.random.default_rng(2)
        rows = np.unique(np.concatenate([[0, wl.T_norm - 1],
                                         rng.choice(wl.T_norm, 512, replace=False)]))
    _rms_check(x, r, w, rows, name)


@pytest.mark.parametrize("C", [768, 2560, 4096, 5120, 8192, 12288, 1, 7, 1001, 40000])
def test_rmsnorm_sweep(C):
    T = max(3, (1 << 20) // (C * 4)) | 1
    x = W.normal_bf16((T, C), 80 + C, 4)
    r = W.normal_bf16((T, C), 80 + C, 5, std=2.0)
    w = W.normal_bf16((C,), 80 + C, 6, mean=1.0, std=0.316)
    _rms_check(x, r, w, None, f"C={C}")


@pytest.mark.parametrize("C", [256, 1000, 5120])
def test_rmsnorm_special_rows(C):
    # one warp per row (C = 256: full rows; 1000: 4 vectors per lane, the last
    # partial) and one CTA per row (5120)
    x = W.normal_bf16((8, C), 5, 4)
    r = torch.zeros((8, C), dtype=torch.bfloat16)
    x[1] = 0                      # all-zero row: y = 0
    x[2] = 1e30                   # squares overflow fp32: double re-sum
    x[3] *= 1e-30                 # squares underflow: double re-sum
    x[4, 5] = float("nan")        # NaN row
    x[5, 7] = float("inf")        # inf row
    x[6] = 3.0                    # constant row
    x[7] *= 2.0 ** -130           # subnormal inputs
    w = W.normal_bf16((C,), 5, 6, mean=1.0, std=0.316)
    _rms_check(x, r, w, None, "special rows")


# Rows of at most 160 vectors of 8 take the one-warp-per-row kernel with 1-5
# vectors per lane (5 without the next-row prefetch), filling the warp or not;
# 1288 is the first width past it.
@pytest.mark.parametrize("C", [136, 264, 512, 520, 1000, 1024, 1032, 1152, 1280, 1288])
def test_rmsnorm_warp_rows(C):
    T = 2053
    x = W.normal_bf16((T, C), 90 + C, 4)
    r = W.normal_bf16((T, C), 90 + C, 5, std=2.0)
    w = W.normal_bf16((C,), 90 + C, 6, mean=1.0, std=0.316)
    _rms_check(x, r, w, None, f"C={C}")


def test_rmsnorm_row_subsets_and_x_is_residual():
    wl = W.WORKLOADS["tiny"]
    x, r, w = W.rmsnorm_inputs(wl)
    yd_full = dt.rmsnorm_residual(to_dev(x), to_dev(r.clone()), to_dev(w), EPS)
    for a, b in [(0, 1), (3, 17), (100, 256)]:
        ys = dt.rmsnorm_residual(to_dev(x[a:b]), to_dev(r[a:b].clone()), to_dev(w), EPS)
        assert_bitexact(bits(ys), bits(yd_full)[a:b], f"rows {a}:{b}")
    # x and residual the same buffer
    xr = to_dev(r.clone())
    y = dt.rmsnorm_residual(xr, xr, to_dev(w), EPS)
    h_exp, y_exp = oracle.rmsnorm_residual(bits(r), bits(r), bits(w), EPS)
    assert_bitexact(bits(xr), h_exp, "x is residual: h")
    assert_within_tolerance(bits(y), y_exp, "x is residual: y")


def test_rmsnorm_misaligned_generic_path():
    T, C = 33, 512
    x = W.normal_bf16((T, C + 1), 3, 4)
    r = W.normal_bf16((T, C + 1), 3, 5, std=2.0)
    w = W.normal_bf16((C + 1,), 3, 6, mean=1.0, std=0.316)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    y = dt.rmsnorm_residual(xd[:, 1:], rd[:, 1:], wd[1:], EPS)
    h_exp, y_exp = oracle.rmsnorm_residual(bits(x)[:, 1:], bits(r)[:, 1:], bits(w)[1:], EPS)
    assert_bitexact(bits(rd)[:, 1:], h_exp, "misaligned h")
    assert_within_tolerance(bits(y), y_exp, "misaligned y")


def test_rmsnorm_empty():
    z = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    assert dt.rmsnorm_residual(z, z.clone(), w).shape == (0, 64)


# ---------------------------------------------------------------- misc

def test_status_errors_raise():
    x = torch.zeros((1, 4, 2, 8), dtype=torch.bfloat16, device=DEV)
    c = torch.zeros((4, 6), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dt.DtrotError):
        dt.rope_rotate_half(x, c[:, :5].contiguous(), c[:, :5].contiguous())  # odd rot_dim


def test_work_is_enqueued_on_the_current_stream():
    wl = W.WORKLOADS["tiny"]
    x = to_dev(W.rope_inputs(wl, "q"))
    freqs = to_dev(W.freqs_for(wl))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c, sn = dt.rope_cos_sin_precompute(freqs)
        out = dt.rope_rotate_half(x, c, sn)
    s.synchronize()
    cos_b, sin_b = oracle.rope_cos_sin(W.freqs_for(wl).numpy())
    assert_bitexact(bits(out), oracle.rope_rotate_half(bits(x), cos_b, sin_b), "side stream")


# ---------------------------------------------------------------- beyond 2^31 elements

def _device_normal(shape, seed, std=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=DEV) * std).to(torch.bfloat16)


def _sample_rows(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rng.choice(n, k, replace=False)]))


def test_geglu_beyond_2_31_elements():
    T, F = 163841, 13200                       # T * F > 2^31, F % 8 == 0
    gu = _device_normal((T, 2 * F), 1)
    out = dt.gelu_and_mul_fused(gu)
    torch.cuda.synchronize()
    rows = _sample_rows(T, 16, 1)
    r = torch.from_numpy(rows).to(DEV)
    g = bits(gu[r])
    assert_bitexact(bits(out[r]), oracle.gelu_and_mul(g[:, :F], g[:, F:]), "2^31+ GEGLU")
    del gu, out


def test_rmsnorm_beyond_2_31_elements():
    T, C = 419431, 5120                        # T * C > 2^31
    x = _device_normal((T, C), 2)
    r = _device_normal((T, C), 3, std=2.0)
    w = _device_normal((C,), 4, std=0.316) + 1.0
    w = w.to(torch.bfloat16)
    rows = _sample_rows(T, 16, 2)
    idx = torch.from_numpy(rows).to(DEV)
    x0, r0 = bits(x[idx]), bits(r[idx])
    y = dt.rmsnorm_residual(x, r, w, EPS)
    torch.cuda.synchronize()
    h_exp, y_exp = oracle.rmsnorm_residual(x0, r0, bits(w), EPS)
    assert_bitexact(bits(r[idx]), h_exp, "2^31+ residual")
    assert_within_tolerance(bits(y[idx]), y_exp, "2^31+ rmsnorm")
    del x, r, y


def test_rope_beyond_2_31_elements():
    B, S, H, D = 1, 32760, 512, 128            # 2.15e9 elements
    x = _device_normal((B, S, H, D), 5)
    freqs = W.freqs_1d(S, B, D)
    c, s = dt.rope_cos_sin_precompute(to_dev(freqs))
    out = dt.rope_rotate_half(x, c, s)
    torch.cuda.synchronize()
    toks = _sample_rows(S, 16, 3)
    t = torch.from_numpy(toks).to(DEV)
    cb, sb = bits(c[t]), bits(s[t])
    assert_bitexact(bits(out[:, t]), oracle.rope_rotate_half(bits(x[:, t]), cb, sb), "2^31+ rope")
    del x, out


# ---------------------------------------------------------------- row subsets, canaries

def test_geglu_and_rope_row_subsets_equal_the_full_run():
    wl = W.WORKLOADS["image"]
    gu = to_dev(W.geglu_inputs(wl))
    full = dt.gelu_and_mul_fused(gu)
    for a, b in [(0, 1), (17, 530), (4000, 4096)]:
        part = dt.gelu_and_mul_fused(gu[a:b].contiguous())
        assert torch.equal(part.view(torch.int16), full[a:b].view(torch.int16)), (a, b)
    x = to_dev(W.rope_inputs(wl, "q"))
    c, s = dt.rope_cos_sin_precompute(to_dev(W.freqs_for(wl)))
    full = dt.rope_rotate_half(x, c, s)
    for a, b in [(0, 1), (333, 1000), (4095, 4096)]:
        part = dt.rope_rotate_half(x[:, a:b], c[a:b].contiguous(), s[a:b].contiguous())
        assert torch.equal(part.view(torch.int16), full[:, a:b].view(torch.int16)), (a, b)


CANARY = 0x7E7E  # a bf16 pattern no op writes here by chance


def _canvas(shape, pad):
    """A buffer with `pad` canary columns on each side of the last dimension and
    one canary row before and after; returns (buffer, the inner view)."""
    *lead, n = shape
    buf = torch.full((*lead[:-1], lead[-1] + 2, n + 2 * pad) if lead else (n + 2 * pad,), 0,
                     dtype=torch.int16, device=DEV)
    buf.fill_(CANARY)
    buf = buf.view(torch.bfloat16)
    inner = buf[..., 1:-1, pad:pad + n] if lead else buf[pad:pad + n]
    return buf, inner


def _canary_intact(buf, inner):
    b = buf.view(torch.int16).clone()
    mask = torch.ones_like(b, dtype=torch.bool)
    if inner.dim() == buf.dim():
        idx = [slice(None)] * (buf.dim() - 2) + [slice(1, -1), slice(None)]
        m2 = torch.zeros_like(mask)
        m2[tuple(idx)] = True
        pad = (buf.shape[-1] - inner.shape[-1]) // 2
        m3 = torch.zeros_like(mask)
        m3[..., pad:pad + inner.shape[-1]] = True
        mask = ~(m2 & m3)
    return bool((b[mask] == CANARY).all())


@pytest.mark.parametrize("pad", [8, 1])
def test_outputs_write_nothing_outside_their_views(pad):
    wl = W.WORKLOADS["tiny"]
    # RoPE out-of-place into a padded (B, S, H, D) view
    x = to_dev(W.rope_inputs(wl, "q"))
    c, s = dt.rope_cos_sin_precompute(to_dev(W.freqs_for(wl)))
    buf, out = _canvas(tuple(x.shape), pad)
    dt.rope_rotate_half(x, c, s, out=out)
    torch.cuda.synchronize()
    assert _canary_intact(buf, out), "rope"
    assert torch.equal(out.view(torch.int16), dt.rope_rotate_half(x, c, s).view(torch.int16))
    # GEGLU into a padded (T, F) view
    gu = to_dev(W.geglu_inputs(wl))
    F = wl.F
    buf, out = _canvas((wl.T_ff, F), pad)
    dt.gelu_and_mul(gu[:, :F], gu[:, F:], out=out)
    torch.cuda.synchronize()
    assert _canary_intact(buf, out), "geglu"
    # RMSNorm: padded out and a padded residual (updated in place)
    xn, r, w = (to_dev(t) for t in W.rmsnorm_inputs(wl))
    rbuf, rv = _canvas(tuple(r.shape), pad)
    rv.copy_(r)
    obuf, ov = _canvas(tuple(xn.shape), pad)
    dt.rmsnorm_residual(xn, rv, w, EPS, out=ov)
    torch.cuda.synchronize()
    assert _canary_intact(rbuf, rv) and _canary_intact(obuf, ov), "rmsnorm"
    # tables: contiguous outputs with canaries before and after
    n = wl.tokens * wl.rot
    cb = torch.full((n + 2 * pad,), CANARY, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    sb = torch.full((n + 2 * pad,), CANARY, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    dt.rope_cos_sin_precompute(to_dev(W.freqs_for(wl)), cb[pad:pad + n].view(wl.tokens, wl.rot),
                               sb[pad:pad + n].view(wl.tokens, wl.rot))
    torch.cuda.synchronize()
    for t in (cb, sb):
        v = t.view(torch.int16)
        assert bool((v[:pad] == CANARY).all() and (v[pad + n:] == CANARY).all()), "tables"


# ---------------------------------------------------------------- launch order

def test_back_to_back_calls_keep_stream_order():
    # Each launch may be scheduled while the previous one drains (programmatic
    # dependent launch); every kernel waits for its predecessor before touching
    # memory.  Queued without synchronisation: table kernels that overwrite the
    # tables the previous RoPE call is reading, RoPE reading them right after, and
    # RMSNorm calls chained through the residual they update in place.
    wl = W.WORKLOADS["image"]
    base = W.freqs_for(wl)
    freqs = [base, base * 0.5 + 0.25, base * 2.0 - 1.0]
    q = W.normal_bf16((wl.B, wl.S, wl.H, wl.D), 11, 0)
    qd = to_dev(q)
    cos = torch.empty((wl.B * wl.S, wl.rot), dtype=torch.bfloat16, device="cuda")
    sin = torch.empty_like(cos)
    outs = []
    for f in freqs:
        dt.rope_cos_sin_precompute(to_dev(f), cos, sin)
        outs.append(dt.rope_rotate_half(qd, cos, sin))
    T, C = 1024, 2048
    xs = [W.normal_bf16((T, C), 12, k) for k in range(3)]
    r = W.normal_bf16((T, C), 12, 5, std=2.0)
    w = W.normal_bf16((C,), 12, 6, mean=1.0, std=math.sqrt(0.1))
    rd, wd = to_dev(r.clone()), to_dev(w)
    ys = [dt.rmsnorm_residual(to_dev(x), rd, wd, EPS) for x in xs]
    torch.cuda.synchronize()
    for i, f in enumerate(freqs):
        ec, es = oracle.rope_cos_sin(f.numpy())
        assert_bitexact(bits(outs[i]), oracle.rope_rotate_half(bits(q), ec, es), f"rope {i}")
    h = bits(r)
    for i, x in enumerate(xs):
        h, y = oracle.rmsnorm_residual(bits(x), h, bits(w), EPS)
        assert_within_tolerance(bits(ys[i]), y, f"rmsnorm {i}")
    assert_bitexact(bits(rd), h, "residual after three calls")


# ---------------------------------------------------------------- 2^14 elements per op

# The smallest sizes of the shape sweep: grids larger than the work (persistent
# RMSNorm and GEGLU grids with more CTAs than rows, RoPE with fewer token warps
# than SMs), element by element against the oracle.
SMALL = 1 << 14


@pytest.mark.parametrize("C", [768, 2560, 4096, 5120])
def test_rmsnorm_2_14_elements(C):
    T = max(1, SMALL // C)
    x = W.normal_bf16((T, C), 300 + C, 4)
    r = W.normal_bf16((T, C), 300 + C, 5, std=2.0)
    w = W.normal_bf16((C,), 300 + C, 6, mean=1.0, std=0.316)
    _rms_check(x, r, w, None, f"T={T} C={C}")


@pytest.mark.parametrize("F", [768, 2560, 4096, 5120])
def test_geglu_2_14_elements(F):
    T = max(1, SMALL // F)
    gu = W.normal_bf16((T, 2 * F), 310 + F, 2)
    _geglu_check(gu, F, None, f"T={T} F={F}")


@pytest.mark.parametrize("S", [16, 5])
@pytest.mark.parametrize("D,rot", SWEEP)
def test_rope_2_14_elements(D, rot, S):
    B = 1
    H = max(1, SMALL // (S * D))
    x = W.normal_bf16((B, S, H, D), 320 + D + rot + S, 0)
    freqs = W.freqs_1d(S, B, rot)
    cos_b, sin_b = oracle.rope_cos_sin(freqs.numpy())
    got_c, got_s = dt.rope_cos_sin_precompute(to_dev(freqs))
    torch.cuda.synchronize()
    assert_bitexact(bits(got_c), cos_b, "cos")
    assert_bitexact(bits(got_s), sin_b, "sin")
    exp = oracle.rope_rotate_half(bits(x), cos_b, sin_b)
    assert_bitexact(_rope_case(x, cos_b, sin_b), exp, f"S={S} H={H} D={D} rot={rot}")
    for mode in ("tables", "angles"):
        _qk_check(B, S, H, max(1, H // 4), D, rot, freqs, 330 + D + rot + S, mode)


# ---------------------------------------------------------------- degenerate sizes

@pytest.mark.parametrize("B,S,H,D,rot", [(1, 1, 1, 2, 2), (2, 3, 1, 8, 2), (1, 5, 3, 6, 4),
                                         (1, 7, 2, 16, 16), (3, 1, 5, 10, 6)])
def test_rope_smallest_shapes(B, S, H, D, rot):
    # one or two pair columns, heads of 2-16 columns, a single token: the
    # generic and narrow-vector paths, the tables and both q+k modes
    x = W.normal_bf16((B, S, H, D), 400 + D + rot, 0)
    freqs = W.freqs_1d(S, B, rot)
    cos_b, sin_b = oracle.rope_cos_sin(freqs.numpy())
    gc, gs = dt.rope_cos_sin_precompute(to_dev(freqs))
    torch.cuda.synchronize()
    assert_bitexact(bits(gc), cos_b, "cos")
    assert_bitexact(bits(gs), sin_b, "sin")
    exp = oracle.rope_rotate_half(bits(x), cos_b, sin_b)
    assert_bitexact(_rope_case(x, cos_b, sin_b), exp, f"B={B} S={S} H={H} D={D} rot={rot}")
    for mode in ("tables", "angles"):
        _qk_check(B, S, H, 1, D, rot, freqs, 410 + D + rot, mode, layout="separate")


@pytest.mark.parametrize("T,F", [(1, 1), (3, 1), (1, 8), (2, 9), (1, 1001)])
def test_geglu_smallest_shapes(T, F):
    gu = W.normal_bf16((T, 2 * F), 420 + T + F, 2)
    _geglu_check(gu, F, None, f"T={T} F={F}")


@pytest.mark.parametrize("T,C", [(1, 8), (1, 2), (2, 1), (1, 5120), (3, 16)])
def test_rmsnorm_smallest_shapes(T, C):
    x = W.normal_bf16((T, C), 430 + T + C, 4)
    r = W.normal_bf16((T, C), 430 + T + C, 5, std=2.0)
    w = W.normal_bf16((C,), 430 + T + C, 6, mean=1.0, std=0.316)
    _rms_check(x, r, w, None, f"T={T} C={C}")


def test_geglu_table_built_into_a_caller_buffer():
    # gelu_table_build + gelu_and_mul(table=) are the two halves of the
    # self-contained call; every gate value through them against the oracle
    from diffusion_transformer_elementwise_rotate_b300 import _capi
    n = int(_capi.load().dtrot_gelu_and_mul_workspace_bytes())
    buf = torch.full((n,), 0xA5, dtype=torch.uint8, device=DEV)   # stale contents
    dt.gelu_table_build(buf)
    gate = torch.from_numpy(np.arange(1 << 16, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).view(64, 1024)
    up = W.normal_bf16((64, 1024), 440, 3)
    out = dt.gelu_and_mul(to_dev(gate), to_dev(up), table=buf)
    torch.cuda.synchronize()
    assert_bitexact(bits(out), oracle.gelu_and_mul(bits(gate), bits(up)), "table in a buffer")


def test_concurrent_callers_on_their_own_streams():
    # four host threads, each on its own stream, run GEGLU (each stream gets its
    # own workspace), RMSNorm and RoPE at once; the library's per-device caches
    # are filled concurrently.  Every result must match the oracle.
    import threading
    wl = W.WORKLOADS["tiny"]
    freqs = W.freqs_for(wl)
    ec, es = oracle.rope_cos_sin(freqs.numpy())
    cases = []
    for i in range(4):
        gu = W.normal_bf16((257, 2 * 520), 600 + i, 2)
        x = W.normal_bf16((129, 768), 600 + i, 4)
        r = W.normal_bf16((129, 768), 600 + i, 5, std=2.0)
        w = W.normal_bf16((768,), 600 + i, 6, mean=1.0, std=0.316)
        q = W.normal_bf16((1, 256, 4, 64), 600 + i, 0)
        cases.append((gu, x, r, w, q))
    results = [None] * 4
    errors = []
    barrier = threading.Barrier(4)

    def work(i):
        try:
            gu, x, r, w, q = cases[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                dgu, dx, dr, dw, dq = (to_dev(t) for t in (gu, x, r, w, q))
                c, s = dt.rope_cos_sin_precompute(to_dev(freqs))
                barrier.wait()
                for _ in range(5):
                    ff = dt.gelu_and_mul_fused(dgu)
                    rr = dr.clone()
                    y = dt.rmsnorm_residual(dx, rr, dw, EPS)
                    qo = dt.rope_rotate_half(dq, c, s)
            st.synchronize()
            results[i] = (bits(ff), bits(rr), bits(y), bits(qo))
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (gu, x, r, w, q) in enumerate(cases):
        ff, rr, y, qo = results[i]
        g = bits(gu)
        assert_bitexact(ff, oracle.gelu_and_mul(g[:, :520], g[:, 520:]), f"thread {i} geglu")
        h, ye = oracle.rmsnorm_residual(bits(x), bits(r), bits(w), EPS)
        assert_bitexact(rr, h, f"thread {i} residual")
        assert_within_tolerance(y, ye, f"thread {i} rmsnorm")
        assert_bitexact(qo, oracle.rope_rotate_half(bits(q), ec, es), f"thread {i} rope")
