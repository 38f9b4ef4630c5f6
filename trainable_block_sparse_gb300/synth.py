"""Seeded synthetic video-shaped inputs and the named workloads.

This module only draws random numbers and shapes them; it holds none of the
attention arithmetic.  Both the CUDA path's tests/benchmark and the fp64
oracle's tests consume exactly these bits, so the two sides always see the same
bf16 inputs.

Recipe (one (batch, head) slice at a time, raster token order r=(t*H+h)*W+w):

* Q, K, V = bf16( N(0,1) noise + s(t,h,w) ) per channel, where s is a smooth
  3-D field: for each channel d, s_d = sum over four modes m of
  a[m,d] * cos(2*pi*(f_m . (t/T, h/H, w/W)) + phi[m,d]) with integer frequency
  vectors f_m in {0,1,2}^3, a ~ N(0,1), phi ~ U[0, 2*pi); each channel is then
  scaled to RMS = amplitude over the positions.  Q and K share one field, so
  attention is spatially local; V has its own.  This gives the concentrated
  cube-level attention mass that "VSA: Faster Video Diffusion with Trainable
  Sparse Attention" reports (key findings: top-32 covers most of the weight).
* Gates G_c, G_f = bf16(sigmoid(N(0,1))), one per token x channel.
* Upstream gradient dO = bf16(N(0,1)).

Every workload has its own seed; each (tensor, batch, head) slice draws from
its own PCG64 stream keyed on (seed, tensor, batch, head).  A query cube whose
noise must be drawn again (test-side gap enforcement) takes a fresh stream
keyed on (seed, tensor, batch, head, cube, attempt), so the redraw touches
that cube only.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math

import numpy as np
import torch

CUBE_T = CUBE_H = CUBE_W = 4
TILE = CUBE_T * CUBE_H * CUBE_W  # tokens per cube: one 64-token tile


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention layer's shapes and selection rule."""

    name: str
    batch: int
    heads: int
    head_dim: int
    T: int
    H: int
    W: int
    select: str  # "topk" (fixed count) or "mass" (variable count)
    topk: int = 32
    mass: float = 0.9
    kmin: int = 8
    kmax: int = 64
    amplitude: float = 1.0
    seed: int = 20260000
    backward: bool = True

    @property
    def tokens(self) -> int:
        return self.T * self.H * self.W

    @property
    def cubes(self) -> int:
        return self.tokens // TILE

    @property
    def bh(self) -> int:
        return self.batch * self.heads

    @property
    def list_capacity(self) -> int:
        """Slots per query cube in the index lists."""
        return self.topk if self.select == "topk" else self.kmax

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # tiny: latent 8x8x8, 2 heads, D=64, top-2 of 8 cubes
    "tiny": Workload("tiny_8x8x8_b1h2d64_k2", 1, 2, 64, 8, 8, 8, "topk", topk=2,
                     seed=20260000),
    # pretraining ablation latent (16,32,32), K=32 of 256 cubes (87.5% sparse)
    "pretrain": Workload("pretrain_16x32x32_b2h12d64_k32", 2, 12, 64, 16, 32, 32,
                         "topk", topk=32, seed=20260001),
    # Wan-1.3B-shaped inference layer, forward only
    "wan13b": Workload("wan13b_20x32x48_b1h12d128_k32", 1, 12, 128, 20, 32, 48,
                       "topk", topk=32, seed=20260002, backward=False),
    # 720p-shaped layer: 70400 tokens, 1100 cubes, 40 heads
    "p720": Workload("p720_20x44x80_b1h40d128_k32", 1, 40, 128, 20, 44, 80,
                     "topk", topk=32, seed=20260003),
    # dynamic compute: smallest top-ranked set with coarse mass >= 0.9, in [8,64]
    "dynamic": Workload("dynamic_16x32x32_b2h12d64_mass0.9", 2, 12, 64, 16, 32, 32,
                        "mass", mass=0.9, kmin=8, kmax=64, amplitude=1.3,
                        seed=20260004),
}


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """Round an fp32 array to bf16 (round to nearest even) as a CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def smooth_field(rng: np.random.Generator, T: int, H: int, W: int, D: int,
                 amplitude: float, n_modes: int = 4) -> np.ndarray:
    """A smooth [T*H*W, D] fp32 field, each channel scaled to RMS = amplitude."""
    f = rng.integers(0, 3, size=(n_modes, 3))
    a = rng.standard_normal((n_modes, D))
    phi = rng.uniform(0.0, 2.0 * math.pi, size=(n_modes, D))
    t = np.arange(T, dtype=np.float64)[:, None, None] / T
    h = np.arange(H, dtype=np.float64)[None, :, None] / H
    w = np.arange(W, dtype=np.float64)[None, None, :] / W
    theta = np.stack([(2.0 * math.pi * (f[m, 0] * t + f[m, 1] * h + f[m, 2] * w)).reshape(-1)
                      for m in range(n_modes)], axis=1)  # [N, modes]
    # cos(theta + phi) = cos(theta)cos(phi) - sin(theta)sin(phi): one small matmul
    basis = np.concatenate([np.cos(theta), -np.sin(theta)], axis=1)       # [N, 2m]
    coef = np.concatenate([a * np.cos(phi), a * np.sin(phi)], axis=0)     # [2m, D]
    s = basis @ coef
    rms = np.sqrt(np.mean(s * s, axis=0))
    s *= amplitude / np.maximum(rms, 1e-12)
    return s.astype(np.float32)


def raster_rows_of_cube(wl: Workload, cube: int) -> np.ndarray:
    """Raster token indices of the 64 tokens of one cube (any order)."""
    cw = wl.W // CUBE_W
    ch = wl.H // CUBE_H
    ct, rem = divmod(cube, ch * cw)
    chh, cww = divmod(rem, cw)
    t = ct * CUBE_T + np.arange(CUBE_T)[:, None, None]
    h = chh * CUBE_H + np.arange(CUBE_H)[None, :, None]
    w = cww * CUBE_W + np.arange(CUBE_W)[None, None, :]
    return ((t * wl.H + h) * wl.W + w).reshape(-1)


_Q, _K, _V, _GC, _GF, _DO, _FIELD_QK, _FIELD_V = range(8)


def _stream(seed: int, *key: int) -> np.random.Generator:
    """An independent PCG64 stream per (workload seed, tensor, batch, head)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


class Inputs:
    """The seeded tensors of one workload (CPU, bf16, [B, heads, N, D] raster).

    Every (tensor, batch, head) slice is drawn from its own keyed stream, so
    the values do not depend on how many threads generate them.
    """

    def __init__(self, wl: Workload, with_grad: bool | None = None, threads: int = 16):
        self.wl = wl
        if with_grad is None:
            with_grad = wl.backward
        B, Hd, N, D = wl.batch, wl.heads, wl.tokens, wl.head_dim
        slices = [(b, h) for b in range(B) for h in range(Hd)]

        def field(b, h, which):
            return smooth_field(_stream(wl.seed, which, b, h), wl.T, wl.H, wl.W, D, wl.amplitude)

        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            fields = list(ex.map(lambda bh: field(*bh, _FIELD_QK), slices))
            self._qk_field = dict(zip(slices, fields))
            vfields = dict(zip(slices, ex.map(lambda bh: field(*bh, _FIELD_V), slices)))

            def make(tensor, add=None, transform=None):
                out = torch.empty((B, Hd, N, D), dtype=torch.bfloat16)

                def one(bh):
                    b, h = bh
                    x = _stream(wl.seed, tensor, b, h).standard_normal((N, D), dtype=np.float32)
                    if add is not None:
                        x += add[bh]
                    if transform is not None:
                        x = transform(x)
                    out[b, h] = to_bf16(x)

                list(ex.map(one, slices))
                return out

            self.q = make(_Q, self._qk_field)
            self.k = make(_K, self._qk_field)
            self.v = make(_V, vfields)
            self.gc = make(_GC, transform=_sigmoid)
            self.gf = make(_GF, transform=_sigmoid)
            self.do = make(_DO) if with_grad else None
        self.redraws = 0

    def redraw_query_cube(self, b: int, h: int, cube: int, attempt: int) -> None:
        """Draw new noise for the 64 query tokens of one cube, keeping the field."""
        wl = self.wl
        rng = _stream(wl.seed, _Q, b, h, cube, attempt)
        rows = raster_rows_of_cube(wl, cube)
        noise = rng.standard_normal((TILE, wl.head_dim), dtype=np.float32)
        vals = noise + self._qk_field[(b, h)][rows]
        self.q[b, h, torch.from_numpy(rows)] = to_bf16(vals)
        self.redraws += 1


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)
