"""GPU test of gemm_run_noalloc, the entry point for callers that cannot
allocate device memory where they run a GEMM: code inside an allocator or
memory-pool callback (allocating there would re-enter the allocator), code
holding a lock the allocator also takes, or programs that reserve all device
memory up front.  It uses a fixed scratch array inside the library instead of
a plan workspace.

Every call goes through the C ABI.  Each result is compared element by
element with the FP64 oracle and with the planned path (gemm_plan + gemm_run)
on the same inputs, within the parity tolerance used everywhere else:
2e-4 * L_act * sum_k |a_ik b_kj| + 1e-6 (+ one output ulp for 16-bit
outputs), and the NaN guard bands around C must be untouched.  The three
problems run back to back twice, so each call finds the previous one's data
in the shared scratch; the second pass must reproduce the first bit for bit.
This file is named to be collected last.
"""
import ctypes
import gc

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


def _setup_call(stream: int) -> int:
    # M = N = 0: the per-device set-up only (scratch address, kernels loaded)
    ep = g13.Epilogue()._c()
    return g13.lib().gemm_run_noalloc(g13.DTYPES["bf16"], 0, 0, 16, None, 16, None, 16, None, 1,
                                      ctypes.byref(ep), None, None, ctypes.c_float(1.0), stream)


CASES = [
    # row strides of A and B not 16-byte aligned, B base 6 bytes off: both staged in
    # scratch; the tensor-core kernel reads the staged copies
    (Workload("noalloc_bf16", "bf16", 300, 263, 1001, alpha=0.5, residual=True,
              dist_a="uniform", dist_b="uniform", dist_r="uniform"), 0, 3),
    # FP32, K-major B, bias + GELU, A base 4 bytes off, K = 301: enough 128-row tiles for
    # the TMA-fed FFMA kernel (not the small-problem variant), which reads the staged
    # copies of both operands
    (Workload("noalloc_f32", "f32", 1024, 1000, 301, b_layout="nk", bias=True, act="gelu"), 1, 0),
    # K-major B with K > 1024: the tensor-core kernel runs as CTA pairs (half-width B boxes)
    (Workload("noalloc_pair_nk", "bf16", 2048, 2048, 1100, b_layout="nk", dist_a="uniform",
              dist_b="uniform"), 0, 0),
]


def _guarded_c(run: Run):
    """A NaN-filled buffer shaped like the planned run's, and the M x N window in it."""
    w = run.w
    buf = torch.full(run.cbuf.shape, float("nan"), dtype=TORCH_OUT[w.out_dtype], device="cuda")
    return buf, buf[:, 1:1 + w.M, 8:8 + w.N]


def _guard_ok(buf: torch.Tensor, w: Workload) -> bool:
    mask = torch.ones(buf.shape, dtype=torch.bool, device=buf.device)
    mask[:, 1:1 + w.M, 8:8 + w.N] = False
    return bool(torch.isnan(buf[mask].float()).all().item())


def test_noalloc_matches_oracle_and_planned_path_twice_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    assert _setup_call(stream) == 0
    runs = [Run(w, seed=11, a_offset=a_off, b_offset=b_off) for w, a_off, b_off in CASES]
    # the planned path's choices, which the entry point shares (besides stream-K / split-K)
    cfgs = {r.w.name: r.info["config"] for r in runs}
    assert cfgs["noalloc_bf16"].kernel == "tc" and cfgs["noalloc_bf16"].stage_a == 1
    assert cfgs["noalloc_f32"].kernel == "ffma" and cfgs["noalloc_f32"].variant != 2
    assert cfgs["noalloc_f32"].stage_a == 1 and cfgs["noalloc_f32"].stage_b == 1
    assert cfgs["noalloc_pair_nk"].variant == 2
    outs = [[_guarded_c(r) for r in runs] for _ in range(2)]
    gc.collect()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for rep in range(2):                 # two passes of back-to-back calls
        for run, (_, C) in zip(runs, outs[rep]):
            rc = _noalloc_call(run, C, stream)
            assert rc == 0, g13.gemm_strerror(rc)
    torch.cuda.synchronize()
    # after the set-up call, no call took device memory (kernels were loaded up front)
    assert torch.cuda.mem_get_info()[0] >= free_before
    for i, run in enumerate(runs):
        w = run.w
        got = outs[0][i][1].float().cpu().double().numpy()
        again = outs[1][i][1].float().cpu().double().numpy()
        assert np.array_equal(got, again), f"{w.name}: second call differs from the first"
        assert _guard_ok(outs[0][i][0], w) and _guard_ok(outs[1][i][0], w), (
            f"{w.name}: store outside the M x N window")
        _, cref, sabs = run.oracle()
        cref, sabs = cref.reshape(got.shape), sabs.reshape(got.shape)
        tol = tolerance(sabs, cref, w)
        err = np.abs(got - cref)
        assert np.all(err <= tol), (w.name, "vs oracle", float(np.max(err / tol)))
        ref = run.run().result()         # the existing entry point, same inputs
        err = np.abs(got - ref)
        assert np.all(err <= tol), (w.name, "vs gemm_run", float(np.max(err / tol)))


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
