"""Device-side failure detection, without faulting the GPU.

A plan made with GEMM_FLAG_TEST_STALL has its first CTA withhold one operand tile
(the producer skips that TMA load), so the consumers' barrier waits can never
complete.  With a 100 ms per-wait limit each wait gives up, the CTA drains the
copies it did issue, frees its TMEM and exits; the plan's status word then reads
GEMM_ERR_DEVICE_TIMEOUT.  Afterwards the context must still work: a normal plan on
the same inputs gives the right answer.

CTA pairs (cta_group::2, chosen for K > 1024) count both CTAs' copies on the
even CTA's barriers.  Withholding the even CTA's first box (or, with
GEMM_FLAG_TEST_STALL_PEER, the odd CTA's) leaves a stage with one share
missing; every wait of both CTAs runs out, the even producer completes the
missing share, sees every issued copy land, and both CTAs leave through the
pair's exit barrier.
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


PAIR = g13.Config("tc", 128, 256, 64, 6, variant=2)


@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("who", ["even", "odd"])
def test_pair_withheld_tile_times_out_and_context_survives(who, layout):
    w = Workload(f"stall_pair_{who}_{layout}", "bf16", 1024, 1024, 2048, b_layout=layout)
    t = w.make(6)
    ldb = w.N if layout == "kn" else w.K
    flag = g13.FLAG_TEST_STALL if who == "even" else g13.FLAG_TEST_STALL_PEER
    stalled = g13.gemm_plan("bf16", w.M, w.N, w.K, w.K, ldb, w.N,
                            g13.Epilogue(b_layout=layout, flags=flag, timeout_ms=100), PAIR)
    assert stalled.info()["config"].variant == 2
    A, B = t["A"].cuda(), t["B"].cuda()
    C = torch.zeros((w.M, w.N), dtype=torch.float32, device="cuda")
    g13.gemm_run(stalled, A, B, C)
    assert g13.gemm_plan_status(stalled) == -5          # GEMM_ERR_DEVICE_TIMEOUT
    # the context is intact: the same pair kernel without the stall is correct
    run = Run(w, tensors=t, config=PAIR)
    C2 = run.run().result()
    run.check(C2)
    assert g13.gemm_plan_status(run.plan) == 0


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_stream_k_missing_partial_times_out_and_context_survives(layout):
    # Stream-K over 3 CTAs: 8 tiles of 32 K blocks, two waves of whole tiles, then
    # the last two tiles' 64 units split 21 / 21 / 22, so the second CTA's range
    # starts inside the seventh tile, whose finisher (the first CTA) waits for
    # that CTA's partial sums.  With GEMM_FLAG_TEST_STALL_PEER the second CTA
    # withholds its first box: its own waits run out, and so does the first
    # CTA's wait for its tags; both exit and the status reads
    # GEMM_ERR_DEVICE_TIMEOUT.
    cfg = g13.Config("tc", 128, 256, 64, 4, stream_k=1, num_ctas=3)
    w = Workload(f"stall_sk_{layout}", "bf16", 512, 512, 2048, b_layout=layout)
    t = w.make(7)
    ldb = w.N if layout == "kn" else w.K
    stalled = g13.gemm_plan("bf16", w.M, w.N, w.K, w.K, ldb, w.N,
                            g13.Epilogue(b_layout=layout, flags=g13.FLAG_TEST_STALL_PEER,
                                         timeout_ms=100), cfg)
    assert stalled.info()["config"].stream_k == 1
    A, B = t["A"].cuda(), t["B"].cuda()
    C = torch.zeros((w.M, w.N), dtype=torch.float32, device="cuda")
    g13.gemm_run(stalled, A, B, C)
    assert g13.gemm_plan_status(stalled) == -5
    run = Run(w, tensors=t, config=cfg)
    C2 = run.run().result()
    run.check(C2)
    assert g13.gemm_plan_status(run.plan) == 0
