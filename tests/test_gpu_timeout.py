"""Device-side failure detection, without faulting the GPU.

A plan made with GEMM_FLAG_TEST_STALL has its first CTA withhold one operand tile
(the producer skips that TMA load), so the consumers' barrier waits can never
complete.  With a 100 ms per-wait limit each wait gives up, the CTA drains the
copies it did issue, frees its TMEM and exits; the plan's status word then reads
GEMM_ERR_DEVICE_TIMEOUT.  Afterwards the context must still work: a normal plan on
the same inputs gives the right answer.
"""
import numpy as np
import pytest
import torch

import dense_gemm_13_gb300 as g13
from dense_gemm_13_gb300.inputs import Workload
from tests.gpu_check import Run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_13_gb300 import _build
    _build.build()
    g13.load()


@pytest.mark.parametrize("dtype,layout", [("bf16", "nk"), ("bf16", "kn"), ("f32", "kn")])
def test_withheld_tile_times_out_and_context_survives(dtype, layout):
    w = Workload(f"stall_{dtype}_{layout}", dtype, 512, 640, 512, b_layout=layout)
    t = w.make(5)
    ldb = w.N if layout == "kn" else w.K
    stalled = g13.gemm_plan(dtype, w.M, w.N, w.K, w.K, ldb, w.N,
                            g13.Epilogue(b_layout=layout, flags=g13.FLAG_TEST_STALL, timeout_ms=100))
    A, B = t["A"].cuda(), t["B"].cuda()
    C = torch.zeros((w.M, w.N), dtype=torch.float32, device="cuda")
    g13.gemm_run(stalled, A, B, C)
    assert g13.gemm_plan_status(stalled) == -5          # GEMM_ERR_DEVICE_TIMEOUT, sticky
    assert g13.gemm_plan_status(stalled) == -5
    # the context is intact: a normal run is correct
    run = Run(w, tensors=t)
    C2 = run.run().result()
    run.check(C2)
    assert g13.gemm_plan_status(run.plan) == 0
