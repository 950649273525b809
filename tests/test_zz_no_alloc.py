"""GPU test of gemm_run_noalloc, the entry point for callers that cannot
allocate device memory where they run a GEMM (e.g. inside an allocator or
memory-pool callback, or after reserving all device memory up front).  It
uses a fixed scratch array inside the library instead of a plan workspace.

The test calls it through the C ABI and compares each result with the
planned path (gemm_plan + gemm_run) on the same inputs, within the parity
tolerance used everywhere else: 2e-4 * L_act * sum_k |a_ik b_kj| + 1e-6 (+ one
output ulp for 16-bit outputs).  Two different problems run back to back, so
the second finds the first one's data in the shared scratch.  This file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_13_gb300 as g13
from dense_gemm_13_gb300.inputs import Workload
from tests.gpu_check import TORCH_OUT, Run, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_13_gb300 import _build
    _build.build()
    g13.load()


def _noalloc_call(run: Run, C: torch.Tensor, stream: int) -> int:
    w = run.w
    ep = run.plan.epilogue._c()
    lda = run.dA.shape[-1]
    ldb = run.dB.shape[-1]
    return g13.lib().gemm_run_noalloc(
        g13.DTYPES[w.dtype], w.M, w.N, w.K, run.dA.data_ptr(), lda, run.dB.data_ptr(), ldb,
        C.data_ptr(), run.ldc, ctypes.byref(ep),
        run.dbias.data_ptr() if run.dbias is not None else None,
        run.dR.data_ptr() if run.dR is not None else None, ctypes.c_float(w.alpha), stream)


CASES = [
    # row strides of A and B not 16-byte aligned, B base 6 bytes off: both staged in scratch
    (Workload("noalloc_bf16", "bf16", 300, 263, 1001, alpha=0.5, residual=True,
              dist_a="uniform", dist_b="uniform", dist_r="uniform"), 0, 3),
    # FP32, K-major B, bias + GELU, A base 4 bytes off: the FFMA kernel reads staged copies
    (Workload("noalloc_f32", "f32", 130, 70, 301, b_layout="nk", bias=True, act="gelu"), 1, 0),
    # K-major B with K > 1024: the tensor-core kernel runs as CTA pairs (half-width B boxes)
    (Workload("noalloc_pair_nk", "bf16", 2048, 2048, 1100, b_layout="nk", dist_a="uniform",
              dist_b="uniform"), 0, 0),
]


def test_noalloc_matches_planned_path_twice_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    runs, outs = [], []
    for w, a_off, b_off in CASES:
        run = Run(w, seed=11, a_offset=a_off, b_offset=b_off)
        if w.name == "noalloc_pair_nk":
            assert run.info["config"].variant == 2      # the same choice the entry point makes
        C = torch.full(run.cbuf.shape, float("nan"), dtype=TORCH_OUT[w.out_dtype],
                       device="cuda")[:, 1:1 + w.M, 8:8 + w.N]
        rc = _noalloc_call(run, C, stream)
        assert rc == 0, g13.gemm_strerror(rc)
        runs.append(run)
        outs.append(C)
    torch.cuda.synchronize()
    for run, C in zip(runs, outs):
        ref = run.run().result()                      # existing entry point, same inputs
        got = C.float().cpu().double().numpy()
        _, cref, sabs = run.oracle()
        tol = tolerance(sabs.reshape(got.shape), cref.reshape(got.shape), run.w)
        err = np.abs(got - ref)
        assert np.all(err <= tol), (run.w.name, float(np.max(err / tol)))


def test_noalloc_rejects_problems_beyond_its_scratch():
    # A is 6000 x 6001 bf16 with an odd row stride: its aligned copy needs about
    # 72 MB, more than the 64 MiB scratch.
    M, N, K = 6000, 64, 6001
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ep = g13.Epilogue()._c()
    rc = g13.lib().gemm_run_noalloc(g13.DTYPES["bf16"], M, N, K, A.data_ptr(), K, B.data_ptr(), N,
                                    C.data_ptr(), N, ctypes.byref(ep), None, None,
                                    ctypes.c_float(1.0), torch.cuda.current_stream().cuda_stream)
    assert rc == -9 and "64 MiB" in g13.gemm_strerror(rc)
    torch.cuda.synchronize()
    assert bool((C == 0).all())         # nothing ran
