"""Seeded synthetic inputs and the named workloads.

This module is shared by the tests, the benchmark and the smoke check; it
holds no GEMM arithmetic -- only random numbers, rounding of those numbers to
the input element type (round-to-nearest-even, done by numpy / torch type
conversion), and the shapes of the workloads.

Recipe: numpy PCG64 streams, one per tensor, seeded as A: s, B: s+1,
bias: s+2, R: s+3.  Values are drawn in float64, rounded to float32 and then
to the element type.  Distributions follow the workloads the pages discuss:
the FP32 SGEMM at 256^3 (uniform [-1,1], the "CUDA Tile ... GEMM" page,
sec. 5.1) and 4096^3 (the "SGEMM ... 83% of cuBLAS" page, sec. 4.1), the
Transformer shapes of the "CUDA Tile ... GEMM" page, sec. 2 (FFN linears and a
batched per-head QK^T), and a ragged shape sweep.
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def matrix(shape, dist: str, seed: int, dtype: str, std: float = 1.0) -> torch.Tensor:
    """A CPU tensor of `shape` with i.i.d. entries: 'uniform' U[-1,1] or 'normal' N(0,std)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = int(np.prod(shape)) if len(shape) else 1
    if dist == "uniform":
        x = rng.uniform(-1.0, 1.0, n)
    elif dist == "normal":
        x = rng.standard_normal(n) * std
    elif dist == "ints":          # small integers in [-4, 4]: exact in every dtype
        x = rng.integers(-4, 5, n).astype(np.float64)
    elif dist == "ones":
        x = np.ones(n)
    else:
        raise ValueError(dist)
    t = torch.from_numpy(x.astype(np.float32).reshape(shape))
    return t.to(TORCH_DTYPES[dtype]).contiguous()


def host_view(t: torch.Tensor) -> np.ndarray:
    """numpy view of a CPU tensor in the form the oracle reads (bf16 as uint16 bits)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@dataclass
class Workload:
    """One GEMM problem: shapes, element types, epilogue and input recipe."""
    name: str
    dtype: str                 # input element type: f32 | f16 | bf16
    M: int
    N: int
    K: int
    batch: int = 1
    b_layout: str = "kn"       # kn: B[K,N] row-major;  nk: B[N,K] row-major (W^T)
    out_dtype: str = "f32"
    alpha: float = 1.0
    beta: float = 1.0
    act: str = "none"
    bias: bool = False
    residual: bool = False
    dist_a: str = "normal"
    dist_b: str = "normal"
    std_a: float = 1.0
    std_b: float = 1.0
    dist_bias: str = "normal"
    std_bias: float = 0.02
    dist_r: str = "normal"
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K * self.batch

    def algorithmic_bytes(self) -> int:
        """Each operand read once, C written once, bias / residual read once."""
        e = {"f32": 4, "f16": 2, "bf16": 2}
        b = self.batch * (self.M * self.K + self.K * self.N) * e[self.dtype]
        b += self.batch * self.M * self.N * e[self.out_dtype]
        if self.bias:
            b += self.N * 4
        if self.residual:
            b += self.batch * self.M * self.N * 4
        return b

    def make(self, seed: int = 0) -> dict:
        """CPU tensors A, B (+ bias, R) for this workload."""
        shp_a = (self.M, self.K) if self.batch == 1 else (self.batch, self.M, self.K)
        kb = (self.K, self.N) if self.b_layout == "kn" else (self.N, self.K)
        shp_b = kb if self.batch == 1 else (self.batch,) + kb
        out = {
            "A": matrix(shp_a, self.dist_a, seed, self.dtype, self.std_a),
            "B": matrix(shp_b, self.dist_b, seed + 1, self.dtype, self.std_b),
            "bias": None,
            "R": None,
        }
        if self.bias:
            out["bias"] = matrix((self.N,), self.dist_bias, seed + 2, "f32", self.std_bias)
        if self.residual:
            shp_c = (self.M, self.N) if self.batch == 1 else (self.batch, self.M, self.N)
            out["R"] = matrix(shp_c, self.dist_r, seed + 3, "f32")
        return out


def _ffn1(dt):
    return Workload(f"ffn1_{dt}", dt, 4096, 3072, 768, b_layout="nk", out_dtype="bf16",
                    act="gelu", bias=True, std_b=0.02,
                    note="X[4096,768] W[3072,768]^T + bias, GELU, BF16 out")


def _ffn2(dt):
    return Workload(f"ffn2_{dt}", dt, 4096, 768, 3072, b_layout="kn", residual=True,
                    note="[4096,3072] [3072,768] + R[4096,768]")


def _qkt(dt):
    return Workload(f"qkt_{dt}", dt, 512, 512, 64, batch=96, b_layout="nk", alpha=0.125,
                    note="96 heads of Q[512,64] K[512,64]^T / 8")


def _qkt_softmax(dt):
    return Workload(f"qkt_softmax_{dt}", dt, 512, 512, 64, batch=96, b_layout="nk", alpha=0.125,
                    act="softmax", out_dtype="bf16",
                    note="96 heads of softmax(Q[512,64] K[512,64]^T / 8) by rows, BF16 out")


WORKLOADS = {w.name: w for w in [
    Workload("sgemm_256", "f32", 256, 256, 256, dist_a="uniform", dist_b="uniform",
             note="FP32 256^3, U[-1,1], seed 0"),
    Workload("sgemm_4096", "f32", 4096, 4096, 4096, note="FP32 4096^3, N(0,1)"),
    Workload("bf16_4096", "bf16", 4096, 4096, 4096, b_layout="nk",
             note="BF16 4096^3, K-major B, FP32 out"),
    Workload("bf16_8192", "bf16", 8192, 8192, 8192, b_layout="nk",
             note="BF16 8192^3, K-major B, FP32 out"),
    _ffn1("bf16"), _ffn1("f16"), _ffn2("bf16"), _ffn2("f16"), _qkt("bf16"), _qkt("f16"),
    _qkt_softmax("bf16"), _qkt_softmax("f16"),
]}

SWEEP_SIZES = (1, 17, 127, 1000, 3001, 4097, 6144)


def sweep_workload(M: int, N: int, K: int) -> Workload:
    """One triple of the ragged BF16 sweep: C = 0.5 A B + 1.0 R, B row-major [K,N]."""
    return Workload(f"sweep_{M}x{N}x{K}", "bf16", M, N, K, b_layout="kn", alpha=0.5, beta=1.0,
                    residual=True, dist_a="uniform", dist_b="uniform", dist_r="uniform")


def sweep() -> list[Workload]:
    return [sweep_workload(M, N, K) for M, N, K in itertools.product(SWEEP_SIZES, repeat=3)]
