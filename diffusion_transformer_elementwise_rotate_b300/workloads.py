"""Seeded synthetic workloads for the DiT elementwise hot path.

This module only draws inputs: it holds none of the hot path's arithmetic and
is shared by the tests, the benchmark and the smoke check.  Everything is
generated on the host with torch CPU generators, so a CPU checker and the GPU
path see bit-identical inputs.

Shapes follow the layer shapes of image and video diffusion transformers:

  tiny   q/k (1, 256, 4, 64), rot 64, one position axis 0..255;
         GEGLU (256, 2x512); RMSNorm (256, 256).
  image  q/k (1, 4096, 32, 128), rot 96 from a (1, 64, 64) t/h/w grid split
         32/32/32 (32 tail columns pass through); GEGLU (4096, 2x12288);
         RMSNorm (4096, 4096).
  cfg    as image with B = 2 (a cond/uncond pair with identical positions),
         rot 128 split 32/48/48; GEGLU (8192, 2x12288); RMSNorm (8192, 4096).
  video  q/k (1, 32760, 40, 128) from a 21x30x52 t/h/w latent grid, rot 128
         split 44/42/42; GEGLU (32760, 2x13824); RMSNorm (32760, 5120).

Value recipe: q, k, gate, up, x ~ N(0, 1); residual ~ N(0, 4) (sigma 2);
w ~ N(1, 0.1) (sigma sqrt(0.1)); all drawn in fp32 and cast to bf16.
Rotary angles: for axis a of width d_a and index i < d_a/2 the angle is
pos_a * 10000^(-2i/d_a), computed in double and stored as fp32; a token's
half-vector is the concatenation over axes and its row is cat(half, half),
the layout a rotate-half table built from per-axis angles has.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Sequence

import torch

THETA = 10000.0
EPS = 1e-6


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    D: int
    grid: tuple          # (t, h, w) positions; tokens are row-major over it
    split: tuple         # rotary widths per axis, summing to rot
    T_ff: int            # GEGLU rows
    F: int               # GEGLU width (gate and up each)
    T_norm: int          # RMSNorm rows
    C: int               # RMSNorm width
    seed: int

    @property
    def rot(self) -> int:
        return sum(self.split)

    @property
    def tokens(self) -> int:
        return self.B * self.S


WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 4, 64, (256,), (64,), 256, 512, 256, 256, 0),
    "image": Workload("image", 1, 4096, 32, 128, (1, 64, 64), (32, 32, 32),
                      4096, 12288, 4096, 4096, 1),
    "cfg": Workload("cfg", 2, 4096, 32, 128, (1, 64, 64), (32, 48, 48),
                    8192, 12288, 8192, 4096, 2),
    "video": Workload("video", 1, 32760, 40, 128, (21, 30, 52), (44, 42, 42),
                      32760, 13824, 32760, 5120, 3),
}

# per-tensor stream offsets
_OFF = {"q": 0, "k": 1, "gate": 2, "up": 3, "x": 4, "residual": 5, "w": 6, "x2": 7,
        "residual2": 8}

_CHUNK = 1 << 24  # elements per draw; fixed so results never depend on size


def generator(seed: int, stream: int) -> torch.Generator:
    return torch.Generator().manual_seed(seed * 1_000_003 + stream)


def normal_bf16(shape: Sequence[int], seed: int, stream: int, mean: float = 0.0,
                std: float = 1.0, pin: bool = False) -> torch.Tensor:
    """bf16 CPU tensor of N(mean, std^2) draws, deterministic in (seed, stream)."""
    g = generator(seed, stream)
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16, pin_memory=pin)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        v = torch.randn(hi - lo, generator=g, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        if mean != 0.0:
            v.add_(mean)
        out[lo:hi] = v.to(torch.bfloat16)
    return out.view(*shape)


def positions(grid: Sequence[int]) -> torch.Tensor:
    """(N, len(grid)) int64 positions, row-major over the grid."""
    axes = [torch.arange(n, dtype=torch.int64) for n in grid]
    mesh = torch.meshgrid(*axes, indexing="ij")
    return torch.stack([m.reshape(-1) for m in mesh], dim=1)


def rotary_angles(pos: torch.Tensor, split: Sequence[int], theta: float = THETA) -> torch.Tensor:
    """(N, sum(split)) fp32 rotary angles laid out as cat(half, half)."""
    pos = pos.to(torch.float64)
    halves = []
    for a, d in enumerate(split):
        i = torch.arange(d // 2, dtype=torch.float64)
        inv = theta ** (-2.0 * i / d)
        halves.append(pos[:, a:a + 1] * inv[None, :])
    half = torch.cat(halves, dim=1)
    return torch.cat([half, half], dim=1).to(torch.float32)


def freqs_for(wl: Workload) -> torch.Tensor:
    """fp32 (S, B, 1, rot): the rotary angles of every token, identical for every
    batch entry (a cond/uncond pair shares positions)."""
    pos = positions(wl.grid)
    if pos.shape[0] != wl.S:
        raise ValueError(f"{wl.name}: grid {wl.grid} has {pos.shape[0]} tokens, S={wl.S}")
    ang = rotary_angles(pos, wl.split)
    return ang[:, None, None, :].expand(wl.S, wl.B, 1, wl.rot).contiguous()


def freqs_1d(S: int, B: int, rot: int) -> torch.Tensor:
    """One position axis 0..S-1 over the whole rotary width."""
    pos = torch.arange(S, dtype=torch.int64)[:, None]
    ang = rotary_angles(pos, (rot,))
    return ang[:, None, None, :].expand(S, B, 1, rot).contiguous()


def rope_inputs(wl: Workload, which: str = "q", pin: bool = False) -> torch.Tensor:
    return normal_bf16((wl.B, wl.S, wl.H, wl.D), wl.seed, _OFF[which], pin=pin)


def geglu_inputs(wl: Workload, pin: bool = False) -> torch.Tensor:
    """One (T, 2F) gate_up buffer: gate = columns [0, F), up = [F, 2F)."""
    T, F = wl.T_ff, wl.F
    gate = normal_bf16((T, F), wl.seed, _OFF["gate"])
    up = normal_bf16((T, F), wl.seed, _OFF["up"])
    out = torch.empty((T, 2 * F), dtype=torch.bfloat16, pin_memory=pin)
    out[:, :F] = gate
    out[:, F:] = up
    return out


def rmsnorm_inputs(wl: Workload, second: bool = False, pin: bool = False):
    """(x, residual, w) for one RMSNorm+residual call; ``second`` draws the
    pre-FFN norm's tensors (the attention norm uses the first set)."""
    T, C = wl.T_norm, wl.C
    x = normal_bf16((T, C), wl.seed, _OFF["x2" if second else "x"], pin=pin)
    r = normal_bf16((T, C), wl.seed, _OFF["residual2" if second else "residual"], std=2.0,
                    pin=pin)
    w = normal_bf16((C,), wl.seed, _OFF["w"], mean=1.0, std=math.sqrt(0.1), pin=pin)
    return x, r, w


def shard_rows(n: int, rank: int, world: int) -> tuple:
    """Contiguous [lo, hi) slice of n token rows owned by `rank` of `world`
    (sizes differ by at most one row).  Every op on this path is per token, so
    shards need no exchange."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


# the GEGLU activation table: one bf16 entry per bf16 gate value
GELU_TABLE_BYTES = 2 * 65536


def algorithmic_bytes(wl: Workload) -> dict:
    """Bytes each op must move at minimum (read inputs once, write outputs once)."""
    return {
        "gelu_table_build": GELU_TABLE_BYTES,
        "rope_cos_sin_precompute": wl.tokens * wl.rot * (4 + 2 + 2),
        "rope_rotate_half": 4 * wl.tokens * wl.H * wl.D + 4 * wl.tokens * wl.rot,
        # q and k in one out-of-place launch: the tables are read once for both
        "rope_rotate_half_qk": 8 * wl.tokens * wl.H * wl.D + 4 * wl.tokens * wl.rot,
        "gelu_and_mul": 6 * wl.T_ff * wl.F,
        "rmsnorm_residual": 8 * wl.T_norm * wl.C + 2 * wl.C,
    }
