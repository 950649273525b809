"""GPU parity: the library (through the C ABI) against the FP64 oracle.

Small problems are compared element by element in full.  The full-size
workloads are compared element by element on every column of a set of rows
and every row of a set of columns: the tile-edge rows and columns plus one at
a random offset inside every 128-wide block, so every output tile (and every
raster-group wrap and persistent wave) has checked elements; a Freivalds
whole-matrix check adds a test for NaNs and gross errors.
Every run also checks the NaN guard bands around C.
"""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_13_gb300 as g13
from dense_gemm_13_gb300.inputs import WORKLOADS, Workload, matrix
from tests.gpu_check import Run, tile_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_13_gb300 import _build
    _build.build()
    g13.load()


def full_check(run: Run):
    C = run.run().result()
    run.check(C)
    assert run.guard_ok(), "store outside the M x N window"
    return C


# ---------------------------------------------------------------- exact integer cases
# Inputs in [-4, 4]: every product and partial sum is an integer below 2^24, so
# FP32 accumulation is exact in any order and the result must equal the oracle.
INT_SHAPES = [(128, 128, 64), (200, 300, 130), (129, 257, 65), (17, 33, 100), (1, 50, 70),
              (300, 7, 90), (256, 512, 1024), (64, 1000, 8), (513, 129, 200)]


def _int_workload(dtype, layout, M, N, K):
    return Workload(f"int_{dtype}_{layout}_{M}x{N}x{K}", dtype, M, N, K, b_layout=layout,
                    dist_a="ints", dist_b="ints")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", INT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_integer(dtype, layout, shape):
    w = _int_workload(dtype, layout, *shape)
    run = Run(w)
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), (
        f"{w.name}: {np.sum(C != cref.reshape(C.shape))} mismatches, config {run.info['config']}")
    assert run.guard_ok()


TC_CONFIGS = [g13.Config("tc", 128, 256, 64, 4), g13.Config("tc", 128, 256, 64, 3),
              g13.Config("tc", 128, 128, 64, 6), g13.Config("tc", 128, 128, 64, 4),
              g13.Config("tc", 128, 256, 64, 3, variant=1),
              g13.Config("tc", 128, 128, 64, 4, variant=1),
              # CTA pairs (tcgen05 cta_group::2) on 256 x 256 tiles
              g13.Config("tc", 128, 256, 64, 6, variant=2),
              g13.Config("tc", 128, 256, 64, 4, variant=2),
              # CTA pairs with eight epilogue warps (C rows TMA cannot store)
              g13.Config("tc", 128, 256, 64, 5, variant=3)]


@pytest.mark.parametrize("cfg", TC_CONFIGS, ids=lambda c: f"bn{c.bn}s{c.stages}v{c.variant}")
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_tc_variants_exact(cfg, dtype, layout):
    # 3 x 3 tiles of 128 x 256 with ragged edges; 5 K blocks with a ragged tail
    w = _int_workload(dtype, layout, 300, 600, 300)
    run = Run(w, config=cfg)
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{w.name} {cfg}"
    assert run.guard_ok()
    # persistent grid smaller than the tile count: each CTA walks several tiles
    cfg2 = g13.Config(cfg.kernel, cfg.bm, cfg.bn, cfg.bk, cfg.stages, num_ctas=2,
                      variant=cfg.variant)
    run2 = Run(w, tensors=run.t, config=cfg2)
    C2 = run2.run().result()
    assert np.array_equal(C2, cref.reshape(C.shape)), f"{w.name} {cfg2} (2 CTAs)"


def test_tc_pair_epilogue_batched():
    # CTA-pair kernel: 3 x 3 pair tiles per batch with ragged edges, every
    # epilogue step, BF16 output through the TMA store path and an odd ldc
    for layout in ("kn", "nk"):
        w = Workload(f"tc_pair_epi_{layout}", "bf16", 700, 520, 1000, batch=2, b_layout=layout,
                     bias=True, act="gelu", residual=True, beta=0.5, alpha=0.25,
                     out_dtype="bf16")
        full_check(Run(w, config=g13.Config("tc", 128, 256, 64, 6, variant=2)))
        full_check(Run(w, config=g13.Config("tc", 128, 256, 64, 4, variant=2), ldc_pad=1))
        full_check(Run(w, config=g13.Config("tc", 128, 256, 64, 5, variant=3), ldc_pad=1))
        full_check(Run(w, config=g13.Config("tc", 128, 256, 64, 5, variant=3)))


RES_CONFIGS = [g13.Config("tc", 128, 256, 64, 3, variant=1, num_ctas=3),
               g13.Config("tc", 128, 128, 64, 6, num_ctas=5),
               g13.Config("tc", 128, 256, 64, 6, variant=2, num_ctas=2)]


@pytest.mark.parametrize("K", [300, 700])
@pytest.mark.parametrize("cfg", RES_CONFIGS, ids=lambda c: f"bn{c.bn}v{c.variant}x{c.num_ctas}")
def test_tc_residual_across_tiles(cfg, K):
    # FP32 residual read by TMA with many tiles per CTA (or pair), ragged M and N:
    # with 5 K blocks the kernel requests each chunk's residual one chunk ahead,
    # also across tile boundaries; with 11 K blocks and several tiles per CTA it
    # reads each chunk's residual when it gets there.
    w = Workload(f"tc_res_{K}", "bf16", 520, 700, K, batch=2, b_layout="nk", bias=True,
                 act="relu", residual=True, alpha=0.5, beta=0.75)
    full_check(Run(w, config=cfg))


SK_CONFIGS = [g13.Config("tc", 128, 256, 64, 4, stream_k=1), g13.Config("tc", 128, 128, 64, 6, stream_k=1),
              g13.Config("tc", 128, 256, 64, 3, variant=1, stream_k=1),
              g13.Config("tc", 128, 256, 64, 6, variant=2, stream_k=1),
              g13.Config("tc", 128, 256, 64, 5, variant=3, stream_k=1)]


@pytest.mark.parametrize("num_ctas", [0, 2, 6, 14])
@pytest.mark.parametrize("cfg", SK_CONFIGS, ids=lambda c: f"bn{c.bn}s{c.stages}v{c.variant}")
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_tc_stream_k_exact(cfg, layout, num_ctas):
    # Tensor-core stream-K: 3 x 3 (pairs: 2 x 3) tiles x 16 K blocks, ragged edges,
    # split over 1, 3 or 7 CTAs (pairs) or the whole GPU, where a tile is cut
    # between up to 16 holders.  Integer inputs: exact in any summation order.
    w = _int_workload("bf16", layout, 300, 600, 1000)
    c = g13.Config(cfg.kernel, cfg.bm, cfg.bn, cfg.bk, cfg.stages, variant=cfg.variant,
                   stream_k=1, num_ctas=num_ctas)
    run = Run(w, config=c)
    assert run.info["config"].stream_k == 1 and run.info["workspace_bytes"] > 0
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{c}"
    assert run.guard_ok()
    C2 = run.run().result()  # bit-identical again (fixed order of the partial sums)
    assert np.array_equal(C, C2)
    assert g13.gemm_plan_status(run.plan) == 0


@pytest.mark.parametrize("cfg", SK_CONFIGS, ids=lambda c: f"bn{c.bn}s{c.stages}v{c.variant}")
def test_tc_stream_k_epilogue_batched(cfg):
    # every epilogue step on a finisher's sum of partials, BF16 out through TMA
    # stores (and, with an odd ldc, the per-row store path), two batches
    w = Workload("tc_sk_epi", "bf16", 700, 520, 1500, batch=2, b_layout="nk", bias=True,
                 act="gelu", residual=True, beta=0.5, alpha=0.25, out_dtype="bf16")
    c = g13.Config(cfg.kernel, cfg.bm, cfg.bn, cfg.bk, cfg.stages, variant=cfg.variant,
                   stream_k=1, num_ctas=10)
    full_check(Run(w, config=c))
    full_check(Run(w, config=c, ldc_pad=1))
    # FP32 out with the residual read by TMA
    w2 = Workload("tc_sk_res", "f16", 520, 700, 1300, b_layout="kn", bias=True, act="relu",
                  residual=True, alpha=0.5, beta=0.75)
    full_check(Run(w2, config=c))


# ---------------------------------------------------------------- 3xTF32 (FP32 on tensor cores)
TF32X3_CONFIGS = [g13.Config("tf32x3", 128, 256, 32, 3, variant=2),
                  g13.Config("tf32x3", 128, 128, 32, 3)]


@pytest.mark.parametrize("cfg", TF32X3_CONFIGS, ids=lambda c: f"bn{c.bn}v{c.variant}")
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", [(300, 600, 300), (513, 129, 200), (17, 33, 101)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32x3_exact_integer(cfg, layout, shape):
    # small integers are TF32 numbers (lo = 0) and every sum is exact in FP32
    w = _int_workload("f32", layout, *shape)
    run = Run(w, config=cfg)
    assert run.info["kernels_per_run"] == 3
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{w.name} {cfg}"
    assert run.guard_ok()
    cfg2 = g13.Config(cfg.kernel, cfg.bm, cfg.bn, cfg.bk, cfg.stages, num_ctas=2, variant=cfg.variant)
    assert np.array_equal(Run(w, tensors=run.t, config=cfg2).run().result(), C)


@pytest.mark.parametrize("cfg", TF32X3_CONFIGS, ids=lambda c: f"bn{c.bn}v{c.variant}")
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_tf32x3_needs_all_three_terms(cfg, layout):
    # x = 1 + 2^-12 is not a TF32 number: hi = 1, lo = 2^-12.  C = K (1 + 2^-12)^2;
    # dropping lo (one TF32 product) errs by 2K * 2^-12 and dropping one cross
    # term by K * 2^-12, both beyond the 2e-4 * sum|ab| tolerance; the three
    # terms leave only lo.lo = K * 2^-24.
    M, N, K = 200, 300, 1000
    x = 1.0 + 2.0 ** -12
    A = torch.full((M, K), x, dtype=torch.float32)
    B = torch.full((K, N) if layout == "kn" else (N, K), x, dtype=torch.float32)
    w = Workload(f"tf32x3_pin_{layout}", "f32", M, N, K, b_layout=layout)
    run = Run(w, tensors={"A": A, "B": B, "bias": None, "R": None}, config=cfg)
    C = run.run().result()
    run.check(C)
    assert np.max(np.abs(C - K * x * x)) <= K * 2.0 ** -20


def test_tf32x3_random_epilogue_batched():
    for layout in ("kn", "nk"):
        w = Workload(f"tf32x3_epi_{layout}", "f32", 700, 520, 1500, batch=2, b_layout=layout,
                     bias=True, act="gelu", residual=True, beta=0.5, alpha=0.25)
        for cfg in TF32X3_CONFIGS:
            full_check(Run(w, config=cfg))
        # shared B across the batch, odd ldc (per-thread epilogue stores)
        t = w.make(3)
        t["B"] = t["B"][0]
        full_check(Run(w, tensors=t, config=TF32X3_CONFIGS[0], ldc_pad=1))


def test_tf32x3_chosen_with_flag_at_4096():
    w = WORKLOADS["sgemm_4096"]
    run = Run(w, flags=g13.FLAG_FP32_TENSOR)
    assert run.info["config"].kernel == "tf32x3"
    C = run.run().result()
    run.check(C, rows=tile_indices(w.M), label=" [rows]")
    run.check(C, cols=tile_indices(w.N), label=" [cols]")
    run.freivalds(C)
    assert Run(w, tensors=run.t).info["config"].kernel == "ffma"   # without the flag: FFMA


@pytest.mark.parametrize("split", [2, 3, 7])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", [(17, 300, 2000), (200, 129, 1500), (1, 64, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tc_split_k_exact(shape, layout, split):
    # K cut into `split` ranges; raw FP32 partial slabs (TMA-stored when N allows,
    # else per-thread) are added in order by a second kernel before the epilogue
    w = _int_workload("bf16", layout, *shape)
    run = Run(w, config=g13.Config("tc", 128, 128, 64, 6, split_k=split))
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{w.name} split {split}"
    assert run.guard_ok()
    assert np.array_equal(C, run.run().result())        # deterministic


def test_tc_split_k_epilogue_batched():
    for layout in ("kn", "nk"):
        w = Workload(f"tc_split_epi_{layout}", "f16", 40, 520, 3000, batch=3, b_layout=layout,
                     bias=True, act="gelu", residual=True, beta=0.5, alpha=0.25, out_dtype="bf16")
        full_check(Run(w, config=g13.Config("tc", 128, 256, 64, 4, split_k=4)))
        full_check(Run(w, config=g13.Config("tc", 128, 256, 64, 3, variant=1, split_k=5)))
    w = Workload("tc_split_auto", "bf16", 17, 6144, 6144, dist_a="uniform", dist_b="uniform",
                 residual=True, dist_r="uniform", alpha=0.5)
    run = Run(w)
    assert run.info["config"].split_k > 1 and run.info["kernels_per_run"] == 2
    C = run.run().result()
    run.check(C, rows=np.arange(17), cols=np.arange(0, 6144, 97))
    run.freivalds(C)


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("stages", [2, 3, 4])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_ffma_variants_exact(bn, variant, stages, layout):
    if bn == 256 and layout == "nk":
        pytest.skip("256-wide FFMA tiles take row-major (KN) B only")
    w = _int_workload("f32", layout, 300, 520, 200)
    run = Run(w, config=g13.Config("ffma", 128, bn, 32, stages, variant=variant))
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape))
    assert run.guard_ok()


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", [(256, 256, 256), (33, 65, 31), (1, 40, 7), (200, 97, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_ffma_small_exact(shape, layout):
    # 32 x 32 tiles from plain loads: ragged tiles and K steps, bit-exact on integers
    w = _int_workload("f32", layout, *shape)
    run = Run(w, config=g13.Config("ffma", 32, 32, 32, 2, variant=2))
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{w.name}"
    assert run.guard_ok()


def test_ffma_small_epilogue_batched_unaligned():
    # every epilogue step, a batch of 3, BF16 output and odd leading dimensions
    # (plain loads: no staging copy, whatever the alignment)
    w = Workload("ffma_small_epi", "f32", 70, 90, 45, batch=3, b_layout="nk", bias=True,
                 act="gelu", residual=True, alpha=0.5, beta=0.25, out_dtype="bf16")
    full_check(Run(w, config=g13.Config("ffma", 32, 32, 32, 2, variant=2), ldc_pad=1))
    w2 = Workload("ffma_small_kn", "f32", 64, 48, 33, b_layout="kn", act="relu", residual=True)
    full_check(Run(w2))  # the dispatcher's choice for a small FP32 problem


@pytest.mark.parametrize("num_ctas", [0, 1, 3, 7, 50])
@pytest.mark.parametrize("bn,variant,layout", [(128, 1, "kn"), (128, 0, "kn"), (128, 0, "nk"),
                                               (256, 1, "kn"), (256, 0, "kn")])
def test_ffma_stream_k_exact(num_ctas, bn, variant, layout):
    # 3 x 3 (or 3 x 2) tiles x 7 K steps spread over a persistent grid; with
    # few CTAs a tile is cut between up to 8 of them and reassembled in order.
    w = _int_workload("f32", layout, 300, 260, 200)
    cfg = g13.Config("ffma", 128, bn, 32, 3, variant=variant, stream_k=1, num_ctas=num_ctas)
    run = Run(w, config=cfg)
    assert run.info["config"].stream_k == 1 and run.info["workspace_bytes"] > 0
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{cfg}"
    assert run.guard_ok()
    # bit-identical on a second run (the partial-sum order is fixed)
    C2 = run.run().result()
    assert np.array_equal(C, C2)


def test_ffma_stream_k_random_batched():
    w = Workload("sk_batched", "f32", 200, 136, 650, batch=3, bias=True, act="relu",
                 residual=True, beta=0.5)
    run = Run(w, config=g13.Config("ffma", 128, 128, 32, 3, variant=1, stream_k=1, num_ctas=5))
    full_check(run)


SKINNY_CASES = [(1, 300, 777, "kn"), (1, 300, 777, "nk"), (300, 1, 777, "kn"), (300, 1, 777, "nk"),
                (5, 333, 1000, "kn"), (5, 333, 1000, "nk"), (333, 3, 500, "kn"), (16, 130, 65, "kn"),
                (17, 90, 333, "kn"), (40, 70, 129, "nk"), (1, 1, 4097, "kn"), (3, 4100, 64, "kn")]


@pytest.mark.parametrize("split", [1, 3, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("case", SKINNY_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}")
def test_skinny_exact(case, dtype, split):
    # the memory-bound kernel in both modes (dot: K-contiguous rows streamed,
    # axpy: N-contiguous columns streamed), with K split over CTAs and the
    # partial sums added in order by a second kernel
    M, N, K, layout = case
    w = _int_workload(dtype, layout, M, N, K)
    run = Run(w, config=g13.Config("skinny", split_k=split))
    assert run.info["kernels_per_run"] == 1
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{w.name} split {split}"
    assert run.guard_ok()
    # the arrival counters were reset: a second run gives the same bits
    assert np.array_equal(run.run().result(), C)


def test_skinny_batched_and_epilogue():
    for layout in ("kn", "nk"):
        w = Workload(f"skinny_b_{layout}", "bf16", 4, 1000, 900, batch=3, b_layout=layout,
                     bias=True, act="gelu", residual=True, beta=0.5, alpha=0.25)
        full_check(Run(w, config=g13.Config("skinny", split_k=4)))
        full_check(Run(w))                                   # dispatcher's choice
    w = Workload("skinny_nsmall", "f32", 700, 2, 3000, batch=2, bias=True, residual=True)
    full_check(Run(w))


# TMA-streamed skinny kernel (variant 1): large-operand rows 16-byte aligned;
# ragged blocks (32 rows for dot, 512 bytes of columns for axpy) and ragged
# K against the stage extent.
SKINNY_TMA_CASES = [(1, 300, 1000, "nk"),   # dot, P = 1
                    (3, 77, 1504, "nk"),    # dot, P = 3 (4-row instantiation)
                    (300, 1, 1000, "kn"),   # N = 1: A streamed, S = B column
                    (200, 4, 1304, "nk"),   # N = 4, S = B rows
                    (200, 3, 1304, "kn"),   # N = 3, S read with a stride of 3
                    (1, 600, 700, "kn"),    # axpy, P = 1
                    (2, 520, 200, "kn"),    # axpy, P = 2
                    (4, 1032, 999, "kn"),   # axpy, P = 4
                    (300, 2, 64, "nk")]     # K shorter than one stage


@pytest.mark.parametrize("num_ctas", [0, 1, 3, 7])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("case", SKINNY_TMA_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}")
def test_skinny_tma_exact(case, dtype, num_ctas):
    # stream-K over the stages: with 3 or 7 CTAs most blocks are cut between
    # CTAs and reassembled from partial sums; with one CTA none is
    M, N, K, layout = case
    w = _int_workload(dtype, layout, M, N, K)
    run = Run(w, config=g13.Config("skinny", variant=1, num_ctas=num_ctas))
    assert run.info["config"].variant == 1 and run.info["kernels_per_run"] == 1
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape)), f"{w.name} {num_ctas} CTAs"
    assert run.guard_ok()
    # the block counters were reset: a second run gives the same bits
    assert np.array_equal(run.run().result(), C)


def test_skinny_tma_batched_epilogue_and_fallback():
    for layout in ("kn", "nk"):
        w = Workload(f"skinny_tma_b_{layout}", "bf16", 4, 1000, 904, batch=3, b_layout=layout,
                     bias=True, act="gelu", residual=True, beta=0.5, alpha=0.25)
        full_check(Run(w, config=g13.Config("skinny", variant=1, num_ctas=5)))
        # one large operand shared by the batch (batch stride 0)
        t = w.make(7)
        t["B"] = t["B"][0]
        full_check(Run(w, tensors=t, config=g13.Config("skinny", variant=1, num_ctas=3)))
    w = Workload("skinny_tma_nsmall", "f32", 700, 2, 3000, batch=2, bias=True, residual=True)
    full_check(Run(w, config=g13.Config("skinny", variant=1, num_ctas=11)))
    full_check(Run(w, config=g13.Config("skinny", variant=1)))
    # the dispatcher's choice for large dot-mode GEMVs is the TMA kernel
    for M, N, layout in ((1, 6144, "nk"), (6144, 1, "kn")):
        w = Workload(f"gemv_{M}x{N}_{layout}", "bf16", M, N, 6144, b_layout=layout,
                     dist_a="uniform", dist_b="uniform")
        run = Run(w)
        assert run.info["config"].kernel == "skinny" and run.info["config"].variant == 1
        full_check(run)
    # a large operand 2 bytes off 16-byte alignment on this run: the plain-load
    # kernel takes over with the same plan, and the answer is the same
    w = Workload("gemv_misaligned", "bf16", 1, 1024, 2048, b_layout="kn", dist_a="ints",
                 dist_b="ints")
    run = Run(w, config=g13.Config("skinny", variant=1), b_offset=1)
    C = run.run().result()
    _, cref, _ = run.oracle()
    assert np.array_equal(C, cref.reshape(C.shape))
    assert run.guard_ok()
    # forcing the TMA kernel on rows TMA cannot address (8194 bytes) is refused
    with pytest.raises(g13.GemmError) as ei:
        g13.gemm_plan("bf16", 1, 4097, 6144, 6144, 4097, 4097, g13.Epilogue(),
                      g13.Config("skinny", variant=1))
    assert ei.value.status == -2


# ---------------------------------------------------------------- epilogues
EPILOGUES = [
    dict(),
    dict(bias=True),
    dict(act="gelu", bias=True),
    dict(act="relu"),
    dict(residual=True, beta=0.5),
    dict(residual=True, bias=True, act="gelu", beta=-1.25),
    dict(out_dtype="bf16", bias=True, act="gelu"),
    dict(out_dtype="f16", residual=True),
]


@pytest.mark.parametrize("epi", EPILOGUES, ids=lambda e: "-".join(f"{k}={v}" for k, v in e.items()) or "plain")
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_epilogue_variants(epi, dtype):
    for layout in ("kn", "nk"):
        w = Workload(f"epi_{dtype}_{layout}", dtype, 333, 520, 200, b_layout=layout, alpha=0.75,
                     **epi)
        full_check(Run(w, seed=3))
        if dtype != "f32":
            # the same epilogue with four epilogue warps (long-K configuration)
            full_check(Run(w, seed=3, config=g13.Config("tc", 128, 256, 64, 4)))
    # the skinny kernel applies the same epilogue
    w = Workload(f"epi_{dtype}_skinny", dtype, 5, 77, 300, alpha=0.75, **epi)
    full_check(Run(w, seed=4))


@pytest.mark.parametrize("epi", [dict(), dict(residual=True, bias=True, act="gelu", beta=-1.25),
                                 dict(out_dtype="bf16", bias=True, act="gelu"),
                                 dict(out_dtype="f16", residual=True)],
                         ids=["plain", "res-bias-gelu", "bf16-gelu", "f16-res"])
@pytest.mark.parametrize("ldc_pad", [1, 3])
def test_epilogue_unaligned_c(epi, ldc_pad):
    # odd row strides of C: the tensor-core epilogue cannot use TMA stores and
    # writes from registers instead; results must be the same
    for layout in ("kn", "nk"):
        w = Workload(f"epi_odd_ldc_{layout}", "bf16", 333, 520, 200, b_layout=layout, alpha=0.75,
                     **epi)
        full_check(Run(w, seed=5, ldc_pad=ldc_pad))


@pytest.mark.parametrize("batch_r", [True, False])
def test_batched_residual_tma(batch_r):
    # batched FP32 residual read by TMA (per-batch R, or one R shared by all entries)
    bt, M, N, K = 4, 200, 264, 136
    A = matrix((bt, M, K), "normal", 0, "bf16")
    B = matrix((bt, K, N), "normal", 1, "bf16")
    R = matrix((bt, M, N) if batch_r else (M, N), "normal", 3, "f32")
    w = Workload("bres", "bf16", M, N, K, batch=bt, residual=True, beta=0.5)
    run = Run(w, tensors={"A": A, "B": B, "bias": None, "R": R})
    if not batch_r:
        run.plan = g13.gemm_plan("bf16", M, N, K, K, N, run.ldc,
                                 g13.Epilogue(residual=True, beta=0.5, ldr=N, batch=bt,
                                              stride_a=M * K, stride_b=K * N,
                                              stride_c=run.cbuf.shape[-1] * run.cbuf.shape[-2],
                                              stride_r=0))
    full_check(run)


# ---------------------------------------------------------------- named workloads
@pytest.mark.parametrize("name", ["sgemm_256", "qkt_bf16", "qkt_f16", "qkt_softmax_bf16",
                                  "qkt_softmax_f16"])
def test_workload_full(name):
    full_check(Run(WORKLOADS[name]))


def test_tc_gelu_pointwise():
    # K = 1 and B = 1 turn the GEMM into GELU(x) on 256 x values in [-8, 8] (exact BF16):
    # the tensor-core epilogue's erf (Abramowitz & Stegun 7.1.26, |error| <= 1.5e-7) must
    # stay within 4e-7 * max(1, |x|) of the FP64 erf form, far inside the GEMM tolerance
    xs = torch.linspace(-8.0, 8.0, 256, dtype=torch.float64).to(torch.bfloat16)
    A = xs.reshape(256, 1).contiguous()
    B = torch.ones((256, 1), dtype=torch.bfloat16)          # NK: B[n][k]
    w = Workload("gelu_points", "bf16", 256, 256, 1, b_layout="nk", act="gelu")
    run = Run(w, tensors={"A": A, "B": B, "bias": None, "R": None})
    assert run.info["config"].kernel == "tc"
    C = run.run().result()
    _, cref, _ = run.oracle()
    x = xs.double().numpy()[:, None]
    assert np.all(np.abs(C - cref.reshape(C.shape)) <= 4e-7 * np.maximum(1.0, np.abs(x)))
    run.check(C)


# ---------------------------------------------------------------- row softmax epilogue
SOFTMAX_CASES = [
    # (M, N, K, layout, bias, out, ldc_pad): N up to 256 runs 256-wide tiles with two TMEM
    # buffers, above that 512-wide tiles (two N = 256 MMAs per K step, one buffer)
    (300, 77, 64, "nk", False, "f32", 0),
    (129, 256, 100, "nk", True, "bf16", 0),
    (200, 257, 64, "kn", True, "f32", 0),
    (513, 512, 72, "nk", False, "bf16", 0),
    (64, 300, 200, "kn", True, "f16", 0),
    (1, 1, 16, "nk", False, "f32", 0),        # a single column: p = 1
    (77, 500, 64, "nk", True, "f32", 1),      # odd ldc: per-thread stores
    (3, 129, 1500, "kn", True, "bf16", 1),
]


@pytest.mark.parametrize("case", SOFTMAX_CASES, ids=lambda c: "x".join(map(str, c[:3])) + c[3])
def test_softmax_rows(case):
    M, N, K, layout, bias, out, pad = case
    w = Workload("softmax_" + "x".join(map(str, case[:3])), "bf16", M, N, K, b_layout=layout,
                 alpha=0.125, bias=bias, act="softmax", out_dtype=out)
    run = Run(w, ldc_pad=pad)
    cfg = run.info["config"]
    assert (cfg.kernel, cfg.bn, cfg.split_k) == ("tc", 256 if N <= 256 else 512, 1)
    C = full_check(run)
    if out == "f32":
        assert np.all(np.abs(C.sum(axis=-1) - 1.0) <= 1e-5)     # each row sums to one
    # persistent grid smaller than the tile count
    cfg2 = g13.Config("tc", 128, cfg.bn, 64, cfg.stages, num_ctas=3, variant=cfg.variant)
    assert np.array_equal(Run(w, tensors=run.t, config=cfg2, ldc_pad=pad).run().result(), C)
    if N <= 256:
        # one thread per whole row (4 epilogue warps, no exchange between warps)
        cfg4 = g13.Config("tc", 128, 256, 64, 4)
        full_check(Run(w, tensors=run.t, config=cfg4, ldc_pad=pad))


def test_softmax_batched_large_logits():
    # 8 heads, alpha = 2 on N(0,1) BF16 inputs with K = 256: logits of size ~30,
    # exp would overflow without the row maximum
    w = Workload("softmax_big", "f16", 256, 384, 256, batch=8, b_layout="nk", alpha=2.0,
                 act="softmax", out_dtype="f32")
    C = full_check(Run(w))
    assert np.all(np.isfinite(C)) and np.all(np.abs(C.sum(axis=-1) - 1.0) <= 1e-5)


@pytest.mark.parametrize("name", ["sgemm_4096", "bf16_4096", "bf16_8192", "ffn1_bf16", "ffn1_f16",
                                  "ffn2_bf16", "ffn2_f16"])
def test_workload_sampled(name):
    w = WORKLOADS[name]
    run = Run(w)
    C = run.run().result()
    rows = tile_indices(w.M)
    cols = tile_indices(w.N)
    assert len(np.unique(rows // 128)) == (w.M + 127) // 128
    assert len(np.unique(cols // 128)) == (w.N + 127) // 128
    run.check(C, rows=rows, label=" [rows: one per 128-row block]")
    run.check(C, cols=cols, label=" [cols: one per 128-column block]")
    if w.act == "none" and w.out_dtype == "f32":
        run.freivalds(C)
    assert run.guard_ok()
    # run-to-run determinism: same inputs, same bits
    C2 = run.run().result()
    assert np.array_equal(C, C2), "result changed between identical runs"


# ---------------------------------------------------------------- edge cases
def test_empty_problems_touch_nothing():
    for M, N in ((0, 64), (64, 0), (0, 0)):
        w = Workload("empty", "bf16", M, N, 64)
        run = Run(w)
        run.run()
        torch.cuda.synchronize()
        assert run.info["kernels_per_run"] == 0
        assert run.guard_ok()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_k_zero_gives_epilogue_of_zero(dtype):
    w = Workload("k0", dtype, 37, 45, 0, bias=True, act="gelu", residual=True, beta=2.0)
    full_check(Run(w))


def test_misaligned_pointers_are_staged_or_rejected():
    # A starts 1 element into its buffer (2-byte aligned): with aligned strides
    # the plan has no workspace and must refuse; with K = 1001 it stages.
    w = Workload("mis", "bf16", 256, 256, 1000)
    with pytest.raises(g13.GemmError) as ei:
        Run(w, a_offset=1).run()
    assert ei.value.status == -3
    w = Workload("mis_staged", "bf16", 256, 263, 1001)     # both row strides misaligned
    run = Run(w, a_offset=1, b_offset=3)
    cfg = run.info["config"]
    assert cfg.stage_a == 1 and cfg.stage_b == 1 and run.info["workspace_bytes"] > 0
    assert run.info["kernels_per_run"] >= 3      # two staging copies + GEMM (+ split reduce)
    full_check(run)
    # FP32 with a misaligned stride goes through the same staging
    w = Workload("mis_staged_f32", "f32", 130, 70, 301, b_layout="nk")
    full_check(Run(w, a_offset=1, b_offset=2))


def test_batched_shared_operand():
    # one B shared by 6 batch entries (stride_b = 0), A and C batched
    bt, M, N, K = 6, 200, 136, 72
    A = matrix((bt, M, K), "normal", 0, "bf16")
    B = matrix((N, K), "normal", 1, "bf16")
    w = Workload("shared_b", "bf16", M, N, K, batch=bt, b_layout="nk")
    run = Run(w, tensors={"A": A, "B": B, "bias": None, "R": None})
    full_check(run)


def test_plan_cache_hits():
    g13.gemm_cache_clear()
    p1 = g13.gemm_plan("bf16", 640, 640, 640, 640, 640, 640)
    p2 = g13.gemm_plan("bf16", 640, 640, 640, 640, 640, 640)
    assert not p1.info()["cache_hit"] and p2.info()["cache_hit"]
    e, h, m = g13.gemm_cache_stats()
    assert (e, h, m) == (1, 1, 1)


def test_invariants_on_gpu():
    # all-ones: every entry equals K exactly
    for dtype, K in (("bf16", 6144), ("f32", 4097), ("f16", 1000)):
        w = Workload("ones", dtype, 300, 260, K, dist_a="ones", dist_b="ones")
        C = Run(w).run().result()
        assert np.all(C == K), (dtype, K)
    # identity: I @ B == B exactly (bf16 B, f32 out)
    n, N = 384, 300
    eye = torch.eye(n).to(torch.bfloat16)
    B = matrix((n, N), "normal", 2, "bf16")
    w = Workload("eye", "bf16", n, N, n)
    C = Run(w, tensors={"A": eye, "B": B, "bias": None, "R": None}).run().result()
    assert np.array_equal(C[0], B.double().numpy())
    # transpose identity: (A B)^T vs B^T A^T through the library, within tolerance of each other
    A = matrix((333, 190), "normal", 3, "bf16")
    Bm = matrix((190, 277), "normal", 4, "bf16")
    w1 = Workload("t1", "bf16", 333, 277, 190)
    w2 = Workload("t2", "bf16", 277, 333, 190)
    r1 = Run(w1, tensors={"A": A, "B": Bm, "bias": None, "R": None})
    r2 = Run(w2, tensors={"A": Bm.t().contiguous(), "B": A.t().contiguous(), "bias": None, "R": None})
    C1, C2 = r1.run().result()[0], r2.run().result()[0]
    _, _, s = r1.oracle()
    assert np.all(np.abs(C1 - C2.T) <= 2 * (2e-4 * s + 1e-6))
