"""Seeded synthetic GroupNorm inputs and the named workloads.

This module holds no GroupNorm arithmetic.  It draws inputs with numpy's PCG64
generator in a fixed order and rounds them to the workload's dtype; both the
CUDA path's tests/bench and the fp64 oracle take their inputs from here.

Recipe (the distributions of the volumetric-UNet GroupNorm sites in the
ScaFFold GroupNorm PRs; activations of a fractal-dataset UNet are not
available, so per-channel Gaussians of the stated spread stand in for them):

  rng = default_rng(seed)
  mu_c  ~ U(-2, 2)      [C]     (+ offset, for the cancellation-probe variant)
  sig_c ~ U(0.5, 3)     [C]     (replaced by 1 in the cancellation-probe variant)
  x[n,c,:] = mu_c + sig_c * z,  z ~ N(0,1) drawn as float32, slab by slab in (n,c) order
  gamma ~ U(0.5, 1.5)   [C]     float32
  beta  ~ N(0, 0.1)     [C]     float32 (sigma 0.1)
  dy[n,c,:] ~ N(0,1)            float32, slab by slab in (n,c) order
  x and dy are then rounded to the dtype (bf16: torch's round-to-nearest-even).

bf16 tensors are returned as uint16 numpy arrays holding the bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32, BF16 = "f32", "bf16"


@dataclass(frozen=True)
class Site:
    """One GroupNorm call: shape (N, C, D, H, W), G groups, dtype, eps."""

    N: int
    C: int
    D: int
    H: int
    W: int
    G: int
    dtype: str = BF16
    eps: float = 1e-5
    mean_offset: float = 0.0
    unit_sigma: bool = False

    @property
    def S(self) -> int:
        return self.D * self.H * self.W

    @property
    def numel(self) -> int:
        return self.N * self.C * self.S

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4

    def min_bytes(self) -> tuple[int, int]:
        """Algorithmic HBM bytes: forward reads x and writes y; backward reads x, dy
        and writes dx (parameters and statistics are not counted)."""
        t = self.numel * self.elem_bytes
        return 2 * t, 3 * t

    def name(self) -> str:
        s = f"{self.dtype} N={self.N} C={self.C} {self.D}x{self.H}x{self.W} G={self.G}"
        if self.mean_offset:
            s += f" offset={self.mean_offset:g}"
        return s


@dataclass
class Workload:
    name: str
    sites: list[Site] = field(default_factory=list)


def _cube(N, C, s, G, dtype=BF16, **kw):
    return Site(N, C, s, s, s, G, dtype, **kw)


# The five workloads: a small fp32 parity case, the 128^3 and 256^3 bf16 volumes
# (ScaFFold problem scales 7 and 8), a many-small-groups case with its large-mean
# cancellation variant, and the UNet encoder/decoder stack of GroupNorm sites.
WORKLOADS = {
    "fp32_2x16x16^3_G4": Workload("fp32_2x16x16^3_G4", [_cube(2, 16, 16, 4, F32)]),
    "bf16_1x32x128^3_G8": Workload("bf16_1x32x128^3_G8", [_cube(1, 32, 128, 8)]),
    "bf16_2x64x96^3_G32": Workload("bf16_2x64x96^3_G32", [_cube(2, 64, 96, 32)]),
    "bf16_2x64x96^3_G32_offset1e3": Workload(
        "bf16_2x64x96^3_G32_offset1e3", [_cube(2, 64, 96, 32, mean_offset=1e3, unit_sigma=True)]),
    "bf16_1x32x256^3_G8": Workload("bf16_1x32x256^3_G8", [_cube(1, 32, 256, 8)]),
    "bf16_unet_stack_G8": Workload(
        "bf16_unet_stack_G8",
        [_cube(1, c, s, 8) for c, s in ((32, 256), (64, 128), (128, 64), (256, 32), (512, 16))]
        + [_cube(1, c, s, 8) for c, s in ((512, 16), (256, 32), (128, 64), (64, 128), (32, 256))]
        + [_cube(1, 48, 97, 8)]),
}


def _to_dtype(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == F32:
        return a32
    import torch  # torch's fp32 -> bf16 conversion (round to nearest even)

    t = torch.from_numpy(a32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def make_inputs(site: Site, seed: int = 0, with_dy: bool = True):
    """Return dict(x, dy, gamma, beta) for `site` (flat NCDHW arrays)."""
    rng = np.random.default_rng(seed)
    C, S, N = site.C, site.S, site.N
    mu = rng.uniform(-2.0, 2.0, C) + site.mean_offset
    sig = rng.uniform(0.5, 3.0, C)
    if site.unit_sigma:
        sig = np.ones(C)
    x32 = np.empty(N * C * S, dtype=np.float32)
    for n in range(N):
        for c in range(C):
            z = rng.standard_normal(S, dtype=np.float32)
            o = (n * C + c) * S
            x32[o:o + S] = np.float32(mu[c]) + np.float32(sig[c]) * z
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = (0.1 * rng.standard_normal(C)).astype(np.float32)
    out = {"x": _to_dtype(x32, site.dtype), "gamma": gamma, "beta": beta}
    del x32
    if with_dy:
        dy32 = np.empty(N * C * S, dtype=np.float32)
        for n in range(N):
            for c in range(C):
                o = (n * C + c) * S
                dy32[o:o + S] = rng.standard_normal(S, dtype=np.float32)
        out["dy"] = _to_dtype(dy32, site.dtype)
    return out


def bits_to_f32(a: np.ndarray) -> np.ndarray:
    """View helper: bf16 bit patterns (uint16) or float32 -> float32 values (exact)."""
    if a.dtype == np.float32:
        return a
    return (a.astype(np.uint32) << 16).view(np.float32)
