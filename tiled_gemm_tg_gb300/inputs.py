"""Seeded synthetic operands for the GEMM workloads.

This module is shared by the tests, the benchmark and the smoke check; it
holds no GEMM arithmetic, only the random draws.  Every operand is drawn in
fp32 on the CPU from ``torch.Generator().manual_seed(seed)`` and then cast to
the input dtype (fp32 -> fp16 rounds to nearest even).  The A seed of a
workload is ``seed_base + 1`` and the B seed ``seed_base + 2``.

The shapes and distributions are the five specified GEMM workloads:
the fp32 128^3 triple-loop example, the fp16 edge set, the A[1024,512] x
B[512,2048] tiling example, the 8192^3 compute-bound square and the two
skinny/wide shapes; two strided batches (256 products of 256^3, 16 of
2048^3); and the 8192^3 square with 8-bit E4M3 inputs.  The pages benchmark on no public dataset, so these
synthetic draws are the whole input set.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str          # "normal", "normal_rsqrtk", "uniform", "normal_0.02", "int2"
    in_dtype: str      # "f16", "f32" or "e4m3"
    out_dtype: str     # "f16" or "f32"
    seed_base: int
    batch: int = 1     # independent products of this shape (a strided batch)

    @property
    def flops(self) -> int:
        return 2 * self.batch * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once (every matrix of the batch)."""
        ein = {"f16": 2, "e4m3": 1}.get(self.in_dtype, 4)
        eout = 2 if self.out_dtype == "f16" else 4
        return self.batch * ((self.M * self.K + self.K * self.N) * ein + self.M * self.N * eout)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("f32_128x128x128", 128, 128, 128, "normal", "f32", "f32", 1000),
        Workload("edge_4x4x4", 4, 4, 4, "normal", "f16", "f16", 2000),
        Workload("edge_128x256x512", 128, 256, 512, "normal", "f16", "f16", 2010),
        Workload("edge_127x255x512", 127, 255, 512, "normal", "f16", "f16", 2020),
        Workload("edge_1x255x17", 1, 255, 17, "normal", "f16", "f16", 2030),
        Workload("tile_1024x2048x512", 1024, 2048, 512, "normal_rsqrtk", "f16", "f16", 3000),
        Workload("square_8192", 8192, 8192, 8192, "uniform", "f16", "f16", 4000),
        Workload("skinny_16x4096x4096", 16, 4096, 4096, "normal_0.02", "f16", "f16", 5000),
        Workload("wide_4096x16384x4096", 4096, 16384, 4096, "normal_0.02", "f16", "f16", 5100),
        # strided batches: many small products in one launch, and a few large ones
        Workload("batched_256x256x256x256", 256, 256, 256, "uniform", "f16", "f16", 6000,
                 batch=256),
        Workload("batched_16x2048x2048x2048", 2048, 2048, 2048, "uniform", "f16", "f16", 6100,
                 batch=16),
        # the 8-bit variant of the compute-bound square: E4M3 in, fp16 out
        Workload("square_8192_e4m3", 8192, 8192, 8192, "uniform", "e4m3", "f16", 7000),
    ]
}

EDGE_SET = ["edge_4x4x4", "edge_128x256x512", "edge_127x255x512", "edge_1x255x17"]


@dataclass(frozen=True)
class AttnWorkload:
    """softmax(scale * Q K^T) V for `batch` independent heads."""
    name: str
    batch: int
    Nq: int
    Nk: int
    d: int
    dv: int
    scale: float
    out_dtype: str     # "f16" or "f32"
    seed_base: int

    @property
    def flops(self) -> int:
        """Q K^T and P V: 2 Nq Nk d + 2 Nq Nk dv per head."""
        return 2 * self.batch * self.Nq * self.Nk * (self.d + self.dv)

    def algorithmic_bytes(self) -> int:
        """Q, K, V read once (fp16), O written once."""
        eout = 2 if self.out_dtype == "f16" else 4
        return self.batch * ((self.Nq * self.d + self.Nk * (self.d + self.dv)) * 2 +
                             self.Nq * self.dv * eout)


ATTN_WORKLOADS = {
    w.name: w
    for w in [
        # the TileLang page's FlashAttention test: one head, seq_len 1024,
        # d_model 768, N(0,1) data, no 1/sqrt(d) factor (fp16 in, fp32 out)
        AttnWorkload("attn_page_1x1024x768", 1, 1024, 1024, 768, 768, 1.0, "f32", 8000),
        # the page's largest length, 2048, as heads of the usual width
        AttnWorkload("attn_16x2048x128", 16, 2048, 2048, 128, 128, 128 ** -0.5, "f16", 8100),
        AttnWorkload("attn_16x4096x128", 16, 4096, 4096, 128, 128, 128 ** -0.5, "f16", 8200),
    ]
}


def attn_operands(w: AttnWorkload):
    """(Q, K, V) fp16 on the CPU, batch x rows x width, N(0,1) draws."""
    q = draw((w.batch, w.Nq, w.d), "normal", w.seed_base + 1, "f16")
    k = draw((w.batch, w.Nk, w.d), "normal", w.seed_base + 2, "f16")
    v = draw((w.batch, w.Nk, w.dv), "normal", w.seed_base + 3, "f16")
    return q, k, v


def draw(shape, dist: str, seed: int, dtype: str, k: int | None = None) -> torch.Tensor:
    """One seeded operand on the CPU, row-major and contiguous."""
    g = torch.Generator().manual_seed(int(seed))
    if dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "normal_rsqrtk":
        if not k:
            raise ValueError("normal_rsqrtk needs the contraction length k")
        x = torch.randn(shape, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(k))
    elif dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal_0.02":
        x = torch.randn(shape, generator=g, dtype=torch.float32) * 0.02
    elif dist == "int2":
        # integers in {-2,...,2}: every product and every partial sum up to
        # 2^24 / 4 terms is exact in fp32, so results are unique.
        x = torch.randint(-2, 3, shape, generator=g).to(torch.float32)
    elif dist == "ones":
        x = torch.ones(shape, dtype=torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist}")
    if dtype == "f16":
        return x.to(torch.float16)
    if dtype == "e4m3":
        # round to nearest even into the 8-bit E4M3 format (|x| stays far
        # below its largest finite value, 448, for every distribution here)
        return x.to(torch.float8_e4m3fn)
    if dtype == "f32":
        return x
    raise ValueError(f"unknown dtype {dtype}")


def operands(w: Workload, dist: str | None = None):
    """(A, B) on the CPU for a workload, from its own seeds: M x K and K x N,
    or batch x M x K and batch x K x N for a strided batch."""
    d = dist or w.dist
    lead = (w.batch,) if w.batch > 1 else ()
    a = draw(lead + (w.M, w.K), d, w.seed_base + 1, w.in_dtype, k=w.K)
    b = draw(lead + (w.K, w.N), d, w.seed_base + 2, w.in_dtype, k=w.K)
    return a, b
