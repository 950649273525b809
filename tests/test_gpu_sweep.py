"""GPU parity over the ragged shape sweep: every (M, N, K) in {1, 17, 127, 1000, 3001,
4097, 6144}^3, BF16 inputs U[-1,1], FP32 residual U[-1,1], C = 0.5 A B + 1.0 R, B row-major [K,N].

Inputs are leading blocks of three seeded 6144 x 6144 matrices (A seed 0, B seed 1,
R seed 3), copied to contiguous tensors, so each triple sees i.i.d. U[-1,1] entries.
Products with M*N*K <= 2^32 are compared in full; larger ones element by element on
every column of the tile-edge rows plus one row inside every 128-row block, and every
row of the same choice of columns (so every output tile has checked elements), plus a
Freivalds whole-matrix check for NaNs and gross errors.  Every run
checks the NaN guard bands and that a second plan of the same shape hits the cache.
"""
import numpy as np
import pytest
import torch

import dense_gemm_13_gb300 as g13
from dense_gemm_13_gb300.inputs import SWEEP_SIZES, matrix, sweep_workload
from tests.gpu_check import Run, tile_indices

pytestmark = pytest.mark.gpu
FULL_LIMIT = 1 << 32
BIG = max(SWEEP_SIZES)


@pytest.fixture(scope="module")
def base():
    from dense_gemm_13_gb300 import _build
    _build.build()
    g13.load()
    return {"A": matrix((BIG, BIG), "uniform", 0, "bf16"),
            "B": matrix((BIG, BIG), "uniform", 1, "bf16"),
            "R": matrix((BIG, BIG), "uniform", 3, "f32")}


@pytest.mark.parametrize("M", SWEEP_SIZES)
def test_sweep(base, M):
    for N in SWEEP_SIZES:
        for K in SWEEP_SIZES:
            w = sweep_workload(M, N, K)
            t = {"A": base["A"][:M, :K].contiguous(), "B": base["B"][:K, :N].contiguous(),
                 "bias": None, "R": base["R"][:M, :N].contiguous()}
            run = Run(w, tensors=t)
            C = run.run().result()
            if M * N * K <= FULL_LIMIT:
                run.check(C)
            else:
                run.check(C, rows=tile_indices(M, seed=1), label=" [rows]")
                run.check(C, cols=tile_indices(N, seed=2), label=" [cols]")
                run.freivalds(C, trials=1)
            assert run.guard_ok(), w.name
            again = g13.gemm_plan("bf16", M, N, K, K, N, run.ldc, run.plan.epilogue)
            assert again.info()["cache_hit"], w.name
            del run, again
        torch.cuda.empty_cache()
