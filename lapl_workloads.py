"""Seeded synthetic workloads for Laplacian-kernel Nystrom attention.

This module holds the workload table and the seeded input generators, nothing else: no step
of the attention method is computed here.  Both the CPU oracle (``oracle/``) and the CUDA
library's tests and benchmark draw their inputs from it, so the two sides see identical values.

Recipe (every workload): ``numpy.random.default_rng(seed)`` (PCG64), seed 0 unless stated;
Q, then K, then V are drawn in that order as float64 arrays of shape [B, H, N, d] (C order),
rounded to float32, and for bf16 workloads rounded again to bfloat16 (round to nearest even).
The returned arrays are float32 whose values are exactly representable in the workload dtype.

Distributions:
  gaussian  Q, K, V ~ N(0, 1)
  student_t Q, K ~ 0.5 * Student-t(df=3) (heavy-tailed query-key L1 distances), V ~ N(0, 1)
  integer   Q, K uniform on {-3, ..., 3}, V ~ N(0, 1)   (distance matrices exact in fp32)
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    grid_h: int
    grid_w: int
    head_dim: int
    num_landmarks: int
    ns_steps: int
    dtype: str            # "f32" or "bf16" (input dtype; outputs are fp32)
    dist: str             # "gaussian" | "student_t" | "integer"
    lam: float = 4.0
    eps: float = 1e-3
    delta: float = 1e-5
    whiten: int = 1
    seed: int = 0

    @property
    def n(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def tokens(self) -> int:
        return self.batch * self.n

    def config(self) -> dict:
        """Scalar configuration as a plain dict (float32-rounded lam/eps/delta)."""
        return dict(batch=self.batch, heads=self.heads, grid_h=self.grid_h, grid_w=self.grid_w,
                    head_dim=self.head_dim, num_landmarks=self.num_landmarks,
                    lam=float(np.float32(self.lam)), eps=float(np.float32(self.eps)),
                    delta=float(np.float32(self.delta)), ns_steps=self.ns_steps,
                    whiten=self.whiten, dtype=self.dtype)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _sweep(n_side: int, dtype: str) -> Workload:
    return Workload(f"sweep_{dtype}_{n_side * n_side}", 1, 8, n_side, n_side, 64, 64, 24, dtype,
                    "gaussian")


WORKLOADS = {w.name: w for w in [
    # tiny: one 16x16 head, 4x4 pooling to 16 landmarks
    Workload("tiny_f32", 1, 1, 16, 16, 32, 16, 20, "f32", "gaussian"),
    Workload("tiny_int", 1, 1, 16, 16, 32, 16, 20, "f32", "integer"),
    # stage-1 vision shape: 56x56 tokens, 8x8 pooling to 49 landmarks, heavy-tailed Q/K
    Workload("stage1_f32", 8, 2, 56, 56, 32, 49, 20, "f32", "student_t"),
    # stage-2/3 vision shape: 28x28 tokens, 4x4 pooling to 49 landmarks, bf16 inputs
    Workload("stage23_bf16", 32, 4, 28, 28, 64, 49, 20, "bf16", "gaussian"),
    # high resolution: 128x128 tokens, 16x16 pooling to 64 landmarks, bf16, heavy-tailed
    Workload("hires_bf16", 4, 8, 128, 128, 64, 64, 24, "bf16", "student_t"),
    # sequence-length sweep, 8x8 landmark grid
    *[_sweep(s, dt) for dt in ("f32", "bf16") for s in (32, 64, 128, 256)],
]}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _draw(rng: np.random.Generator, dist: str, shape, role: str) -> np.ndarray:
    if dist == "gaussian" or role == "v":
        return rng.standard_normal(shape)
    if dist == "student_t":
        return 0.5 * rng.standard_t(3, shape)
    if dist == "integer":
        return rng.integers(-3, 4, size=shape).astype(np.float64)
    raise ValueError(dist)


def make_inputs(w: Workload, seed: int | None = None):
    """Return (q, k, v) as float32 arrays [B,H,N,d], exactly representable in ``w.dtype``."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    shape = (w.batch, w.heads, w.n, w.head_dim)
    out = []
    for role in ("q", "k", "v"):
        a = _draw(rng, w.dist, shape, role).astype(np.float32)
        if w.dtype == "bf16":
            a = round_to_bf16(a)
        out.append(a)
    return tuple(out)


def make_bias(w: Workload, seed: int = 1, scale: float = 0.1) -> np.ndarray:
    """A seeded non-zero bias [H, m] (float32) for exercising the bias path."""
    rng = np.random.default_rng(seed)
    return (scale * rng.standard_normal((w.heads, w.num_landmarks))).astype(np.float32)
