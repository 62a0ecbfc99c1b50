"""Element-wise comparison of bf16 bit arrays (numpy uint16)."""
import numpy as np

# Tolerance for GEGLU and RMSNorm: every element within 1 bf16 ulp,
# and at most 0.01% of elements different at all.  RoPE and the cos/sin tables
# must be bit-exact.
MAX_ULP = 1
MAX_MISMATCH_FRACTION = 1e-4


def _key(u):
    u = u.astype(np.int64)
    return np.where(u & 0x8000, 0x8000 - (u & 0x7FFF), 0x8000 + u)


def is_nan(u):
    return ((u & 0x7F80) == 0x7F80) & ((u & 0x007F) != 0)


def ulp_diff(a, b):
    """Distance in bf16 steps (ordered keys; +0 and -0 are one step apart is
    avoided by mapping both zeros to the same key); NaN == NaN counts as 0."""
    a = np.asarray(a, np.uint16)
    b = np.asarray(b, np.uint16)
    ka, kb = _key(a), _key(b)
    ka = np.where((a & 0x7FFF) == 0, 0x8000, ka)
    kb = np.where((b & 0x7FFF) == 0, 0x8000, kb)
    d = np.abs(ka - kb)
    both_nan = is_nan(a) & is_nan(b)
    one_nan = is_nan(a) ^ is_nan(b)
    d = np.where(both_nan, 0, d)
    return np.where(one_nan, 1 << 20, d)


def assert_bitexact(got, exp, what=""):
    got = np.asarray(got, np.uint16)
    exp = np.asarray(exp, np.uint16)
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    same = (got == exp) | (is_nan(got) & is_nan(exp))
    if not same.all():
        idx = np.argwhere(~same)[:8]
        detail = [(tuple(i), hex(int(got[tuple(i)])), hex(int(exp[tuple(i)]))) for i in idx]
        raise AssertionError(f"{what}: {np.count_nonzero(~same)} of {same.size} differ; "
                             f"first {detail}")


def assert_within_tolerance(got, exp, what=""):
    d = ulp_diff(got, exp)
    n = np.count_nonzero(d)
    assert d.max(initial=0) <= MAX_ULP, f"{what}: max ulp diff {d.max()}"
    assert n <= MAX_MISMATCH_FRACTION * d.size, f"{what}: {n} of {d.size} differ"
    return n
