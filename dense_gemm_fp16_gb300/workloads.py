"""Seeded synthetic inputs for the two products, shared by the tests, the
smoke check and the benchmark.

This module only draws numbers: it holds none of the products' arithmetic and
imports neither the CUDA library nor the oracle.  Every tensor is produced on
the CPU from a ``torch.Generator`` seeded explicitly, so the oracle and the
GPU path always consume the very same host arrays.

The first five named workloads follow the pages' own test and benchmark shapes:

* SGEMM 256³ with A from seed 1 and B from seed 2, values uniform in [-1, 1]
  (the correctness size of the host harness in "异步拷贝与 Hopper/Blackwell
  新特性", section "cp.async 与多级流水 sm_80+"), 1024³, and the 4096³
  benchmark size of the same harness, here with alpha = 1, beta = 0.5 and a
  C drawn from seed 3.
* fp16 NT 5376 × 5376 × 2048, uniform [-1, 1] rounded to half (the problem of
  "从零开始的 AI Infra: 算子基础与GPU架构", section "背景与分析").
* fp16 NT 5000 × 5376 × 2040, normal(0, 1) rounded to half, seeds 4 and 5:
  the same problem with M and K off the tile grid, to exercise the tails.

A sixth, 1 × 16384 × 8192, is a decode-sized matrix-vector product for the
M = 1 path ("第 6 章 · Shared Memory & Tile", section "6.5.5 GEMV (M=1)").
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    form: str            # "sgemm" or "f16_nt"
    M: int
    N: int
    K: int
    dist: str            # "uniform" (in [-1, 1]) or "normal" (mean 0, sd 1)
    seed_a: int
    seed_b: int
    seed_c: Optional[int] = None
    alpha: float = 1.0
    beta: float = 0.0

    @property
    def flop(self) -> int:
        """2·M·N·K, the operation count both pages use for throughput."""
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    w.name: w
    for w in [
        Workload("sgemm_256", "sgemm", 256, 256, 256, "uniform", 1, 2),
        Workload("sgemm_1024", "sgemm", 1024, 1024, 1024, "uniform", 1, 2),
        Workload("sgemm_4096", "sgemm", 4096, 4096, 4096, "uniform", 1, 2, 3, 1.0, 0.5),
        Workload("f16_nt_5376x5376x2048", "f16_nt", 5376, 5376, 2048, "uniform", 1, 2),
        Workload("f16_nt_5000x5376x2040", "f16_nt", 5000, 5376, 2040, "normal", 4, 5),
        # A decode-sized matrix-vector product for the M = 1 path: one row of A
        # against a 256 MB B (not a page workload; it measures that path's HBM
        # roofline).
        Workload("f16_gemv_1x16384x8192", "f16_nt", 1, 16384, 8192, "uniform", 6, 7),
        # The same B against 16 rows of A (a small decode batch): the skinny
        # tensor-core path, also bound by reading B once.
        Workload("f16_skinny_16x16384x8192", "f16_nt", 16, 16384, 8192, "uniform", 8, 7),
        # Few 256 x 256 tiles over a long K (32 tiles, 128 k-blocks): the
        # shape class the K split over two CTA pairs per cluster serves.
        Workload("f16_ksplit_1024x2048x8192", "f16_nt", 1024, 2048, 8192, "uniform", 10, 11),
    ]
}

# The throughput workload: the fp16 NT problem the pages tune.
HEADLINE = "f16_nt_5376x5376x2048"


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw_f32(shape, seed: int, dist: str = "uniform") -> torch.Tensor:
    """A float32 CPU tensor: uniform in [-1, 1] or standard normal."""
    g = _gen(seed)
    if dist == "uniform":
        return torch.rand(tuple(shape), generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def draw_f16(shape, seed: int, dist: str = "uniform") -> torch.Tensor:
    """A half CPU tensor: the float32 draw rounded to nearest half."""
    return draw_f32(shape, seed, dist).to(torch.float16)


def draw_int(shape, seed: int, lo: int, hi: int, dtype=torch.float32) -> torch.Tensor:
    """Integer values in [lo, hi] stored in a float dtype (exact products)."""
    g = _gen(seed)
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int64).to(dtype)


def draw_mxfp8(rows: int, K: int, seed: int, scale_lo: int = 125, scale_hi: int = 129):
    """Block-scaled FP8 operands as stored: E4M3 codes [rows, K] (uint8) and
    UE8M0 scale codes [rows, K/32] (uint8).  Elements are standard-normal
    draws cast to E4M3 by PyTorch; scale codes are uniform integers in
    [scale_lo, scale_hi] (2^-2 .. 2^2 by default)."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    g = _gen(seed)
    x = torch.randn((rows, K), generator=g, dtype=torch.float32)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
    scales = torch.randint(scale_lo, scale_hi + 1, (rows, K // 32), generator=g, dtype=torch.int64)
    return codes.contiguous(), scales.to(torch.uint8).contiguous()


def draw_nvfp4(rows: int, K: int, seed: int):
    """Block-scaled FP4 operands as stored: E2M1 elements packed two per byte
    [rows, K/2] (uint8, uniform random bits: every code equally likely) and
    UE4M3 block scales [rows, K/16] (uint8): values uniform in [0.25, 4]
    cast to E4M3 by PyTorch."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    g = _gen(seed)
    packed = torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.int64).to(torch.uint8)
    sv = torch.rand((rows, K // 16), generator=g, dtype=torch.float32) * 3.75 + 0.25
    scales = sv.to(torch.float8_e4m3fn).view(torch.uint8)
    return packed.contiguous(), scales.contiguous()


def make_inputs(w: Workload):
    """Host tensors (A, B, C0) of a workload; C0 is None when beta == 0."""
    if w.form == "f16_nt":
        A = draw_f16((w.M, w.K), w.seed_a, w.dist)
        B = draw_f16((w.N, w.K), w.seed_b, w.dist)
        return A, B, None
    if w.form == "sgemm":
        A = draw_f32((w.M, w.K), w.seed_a, w.dist)
        B = draw_f32((w.K, w.N), w.seed_b, w.dist)
        C0 = None
        if w.seed_c is not None:
            C0 = draw_f32((w.M, w.N), w.seed_c, w.dist)
        return A, B, C0
    raise ValueError(f"unknown form {w.form!r}")


def sample_positions(M: int, N: int, count: int, seed: int, tail_rows=None):
    """Seeded output positions for a sampled comparison.

    ``count`` distinct (row, col) pairs drawn without replacement from M×N,
    plus forced coverage: the four corners, every element of the last row and
    of the last column, and every column of each row in ``tail_rows``.
    Returns two int64 numpy arrays (rows, cols) without duplicates."""
    import numpy as np

    total = M * N
    rng = np.random.default_rng(seed)
    count = min(count, total)
    flat = rng.choice(total, size=count, replace=False) if count else np.zeros(0, np.int64)
    extra = []
    if M and N:
        extra += [0, N - 1, (M - 1) * N, (M - 1) * N + N - 1]
        extra += list((M - 1) * N + np.arange(N))          # last row
        extra += list(np.arange(M) * N + (N - 1))          # last column
        for r in tail_rows or []:
            if 0 <= r < M:
                extra += list(r * N + np.arange(N))
    flat = np.unique(np.concatenate([flat.astype(np.int64), np.asarray(extra, dtype=np.int64)]))
    return (flat // N).astype(np.int64), (flat % N).astype(np.int64)
