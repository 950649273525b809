"""CPU tests of the C ABI: the library loads, exports every declared symbol,
validates arguments, and the dispatcher picks the expected buckets.  No
kernel runs here (there is no GPU); calls that need a device must say so."""
import ctypes
import os
import re

import pytest

import dense_gemm_13_gb300 as g13
from dense_gemm_13_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm13.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return g13.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(gemm_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("gemm_plan", "gemm_run", "gemm_plan_destroy", "gemm_plan_status", "gemm_strerror"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_strerror_and_version(lib):
    assert g13.gemm_strerror(0) == "ok"
    for code in range(-8, 0):
        assert g13.gemm_strerror(code) not in ("", "unknown status")
    assert g13.gemm_strerror(-99) == "unknown status"
    assert "sm_103a" in g13.gemm_version()


def _rc(lib, dtype=2, M=64, N=64, K=64, lda=64, ldb=64, ldc=64, ep=None):
    h = ctypes.c_void_p()
    e = (ep or g13.Epilogue())._c()
    return lib.gemm_plan(dtype, M, N, K, lda, ldb, ldc, ctypes.byref(e), ctypes.byref(h))


def test_validation_codes(lib):
    E = g13.Epilogue
    bad = [
        dict(M=-1), dict(N=-1), dict(K=-1),
        dict(lda=63), dict(ldb=63), dict(ldc=63),
        dict(dtype=7),
        dict(ep=E(batch=2, stride_c=10)),           # C batches would overlap
        dict(ep=E(residual=True, ldr=32)),          # ldr < N
        dict(ep=E(stride_a=-1)),
    ]
    for kw in bad:
        assert _rc(lib, **kw) == -1, kw
    # bad enum values inside the epilogue
    e = g13.Epilogue()._c()
    e.act = 9
    h = ctypes.c_void_p()
    assert lib.gemm_plan(2, 64, 64, 64, 64, 64, 64, ctypes.byref(e), ctypes.byref(h)) == -1
    e = g13.Epilogue()._c()
    e.out_dtype = 5
    assert lib.gemm_plan(2, 64, 64, 64, 64, 64, 64, ctypes.byref(e), ctypes.byref(h)) == -1
    # NULL out_plan
    assert lib.gemm_plan(2, 64, 64, 64, 64, 64, 64, None, None) == -1
    # NK layout: ldb must cover K, not N
    assert _rc(lib, M=64, N=256, K=32, lda=32, ldb=32, ldc=256, ep=E(b_layout="nk")) in (0, -7)
    assert _rc(lib, M=64, N=256, K=32, lda=32, ldb=31, ldc=256, ep=E(b_layout="nk")) == -1


def test_valid_plan_needs_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _rc(lib) == -7       # GEMM_ERR_NO_DEVICE, not a crash


def test_run_and_status_reject_bad_plans(lib):
    bogus = ctypes.c_void_p(0x1234)
    assert lib.gemm_run(None, None, None, None, None, None, ctypes.c_float(1.0), None) == -6
    assert lib.gemm_run(bogus, None, None, None, None, None, ctypes.c_float(1.0), None) == -6
    assert lib.gemm_plan_status(bogus) == -6
    info = g13._PlanInfo()
    assert lib.gemm_plan_info(bogus, ctypes.byref(info)) == -6
    lib.gemm_plan_destroy(None)     # no-op
    lib.gemm_plan_destroy(bogus)    # unknown handle: ignored


def sel(dtype, M, N, K, layout="kn", sms=152, **kw):
    lda = max(K, 1)
    ldb = max(N if layout == "kn" else K, 1)
    return g13.gemm_select_config(dtype, M, N, K, lda, ldb, max(N, 1),
                                  g13.Epilogue(b_layout=layout, **kw), num_sms=sms)


def test_dispatch_buckets(lib):
    c = sel("f32", 4096, 4096, 4096)
    assert (c.kernel, c.variant, c.bn, c.stream_k) == ("ffma", 1, 256, 1)   # packed, wide, stream-K
    c = sel("f32", 8192, 8192, 8192)
    assert (c.bn, c.stream_k) == (256, 0)               # 2048 tiles = 13.5 waves: whole tiles
    c = sel("f32", 256, 256, 256)
    assert (c.bm, c.bn, c.variant, c.stream_k) == (32, 32, 2, 0)   # 4 tiles: small 32 x 32 tiles
    c = sel("f32", 1024, 1024, 1024)
    assert (c.bn, c.variant, c.stream_k) == (128, 1, 1)  # 64 tiles: stream-K
    assert sel("f32", 4096, 4096, 4096, "nk").variant == 0
    assert sel("f32", 256, 256, 256).kernel == "ffma"
    c = sel("bf16", 8192, 8192, 8192, "nk")
    assert (c.kernel, c.bm, c.bn, c.bk, c.variant, c.stages) == ("tc", 128, 256, 64, 2, 6)  # pairs
    c = sel("f16", 4096, 3072, 768, "nk", bias=True, act="gelu", out_dtype="bf16")
    assert (c.kernel, c.variant, c.stages) == ("tc", 1, 3)   # short K, heavy epilogue: 8 warps
    c = sel("f16", 4096, 3072, 768, "nk")
    assert (c.kernel, c.variant, c.stages) == ("tc", 3, 5)   # main loop outlasts a plain epilogue
    c = sel("bf16", 6144, 6144, 1000, residual=True)
    assert (c.kernel, c.variant, c.stages) == ("tc", 3, 5)   # ... and an FP32 residual
    assert sel("bf16", 6144, 6144, 127, residual=True).variant == 1   # 2 K blocks: epilogue-bound
    assert sel("bf16", 6144, 4097, 1000, residual=True).variant == 1  # rows TMA cannot store
    # the short-K pair rule's epilogue weights: bias + GELU over 16 K blocks still pairs,
    # GELU with a residual never does for K <= 1024, nor one wave of single tiles
    assert sel("bf16", 4096, 4096, 1024, "nk", bias=True, act="gelu").variant == 3
    assert sel("bf16", 4096, 4096, 1024, "nk", bias=True, act="gelu", residual=True).variant == 1
    assert sel("bf16", 4096, 4096, 512, "nk", bias=True).variant == 3
    assert sel("bf16", 4096, 4096, 384, "nk").variant == 1             # 6 K blocks: epilogue-bound
    assert sel("bf16", 4096, 4096, 1024, "nk", sms=1).variant == 1     # a pair needs two SMs
    c = sel("bf16", 4096, 768, 3072, "kn")
    assert (c.kernel, c.variant) == ("tc", 2)                # 48 pair tiles: one wave of pairs
    c = sel("bf16", 256, 256, 4096, "nk")
    assert (c.kernel, c.variant) == ("tc", 0) and c.split_k > 1   # split-K runs single CTAs
    c = sel("bf16", 8192, 8192, 8192, "nk", sms=1)
    assert c.variant not in (2, 3)                           # a pair needs two SMs
    c = sel("bf16", 3001, 3001, 3001)                        # C rows of 12004 bytes: no TMA store
    assert (c.kernel, c.variant, c.stages) == ("tc", 3, 5)   # pairs with eight epilogue warps
    assert sel("bf16", 3001, 3000, 3001).variant == 2        # 12000-byte rows: TMA stores
    for M, N in ((1, 6144), (6144, 1), (0, 10), (10, 0)):
        assert sel("bf16", M, N, 1000).kernel == "skinny", (M, N)
    assert sel("bf16", 512, 512, 0).kernel == "skinny"      # K = 0: epilogue only
    assert sel("f32", 1, 4096, 4096).kernel == "skinny"
    assert sel("bf16", 4, 4096, 4096).kernel == "skinny"
    assert sel("bf16", 5, 4096, 4096).kernel == "tc"       # tensor cores (+ split-K) from 5 rows
    # FP32 on the tensor cores (3xTF32) only when the caller allows it
    c = sel("f32", 4096, 4096, 4096, flags=g13.FLAG_FP32_TENSOR)
    assert (c.kernel, c.bn, c.variant, c.stages, c.stage_a, c.stage_b) == ("tf32x3", 256, 2, 3, 0, 0)
    assert sel("f32", 100, 4096, 4096, flags=g13.FLAG_FP32_TENSOR).bn == 128   # single CTAs
    assert sel("f32", 256, 256, 256, flags=g13.FLAG_FP32_TENSOR).kernel == "ffma"  # too small
    assert sel("bf16", 4096, 4096, 4096, flags=g13.FLAG_FP32_TENSOR).kernel == "tc"


def test_dispatch_skinny_tma(lib):
    # large dot-mode problems (the large operand's rows hold K) with 16-byte-aligned
    # rows stream through the TMA ring (variant 1); axpy mode (B in KN layout with M
    # small), small problems and unaligned rows take the plain-load kernel (variant 0)
    for M, N, K, lay in ((1, 6144, 6144, "nk"), (6144, 1, 6144, "kn"), (6144, 4, 6144, "kn"),
                         (2, 6144, 4096, "nk"), (1000, 1, 6144, "nk")):
        c = sel("bf16", M, N, K, lay)
        assert (c.kernel, c.variant, c.split_k) == ("skinny", 1, 1), (M, N, K, lay)
    for M, N, K, lay in ((1, 6144, 6144, "kn"), (4, 6144, 6144, "kn"), (1, 1000, 1000, "nk"),
                         (6144, 1, 4097, "kn"), (1, 6144, 4097, "nk")):
        assert sel("bf16", M, N, K, lay).variant == 0, (M, N, K, lay)
    # P = 4 rows of K as FP32 beside a 4-stage ring: K = 6144 fits, 16384 does not
    assert sel("bf16", 6144, 4, 6144).variant == 1
    assert sel("bf16", 6144, 4, 16384).variant == 0


def test_dispatch_small_fp32(lib):
    # 32 x 32 tiles from plain loads when the 128 x 128 tiles number at most one per
    # eight SMs and K <= 512; otherwise the TMA-fed kernel (stream-K or whole tiles)
    for M, N, K in ((256, 256, 256), (512, 512, 512), (300, 17, 100), (40, 9, 7)):
        c = sel("f32", M, N, K)
        assert (c.kernel, c.variant, c.bm, c.bn, c.stream_k) == ("ffma", 2, 32, 32, 0), (M, N, K)
        assert (c.stage_a, c.stage_b) == (0, 0)
    assert sel("f32", 512, 512, 1024).variant != 2           # longer K: stream-K splits K
    assert sel("f32", 1024, 1024, 512).variant != 2          # 64 tiles > 152 / 8
    assert sel("f32", 256, 256, 256, batch=96, stride_a=256 * 256, stride_b=256 * 256,
               stride_c=256 * 256).variant != 2             # 384 tiles across the batch
    assert sel("f32", 256, 256, 256, sms=8).variant != 2     # 4 tiles > 8 / 8
    assert sel("bf16", 256, 256, 256).kernel == "tc"        # FP32 only


def test_softmax_limits(lib):
    # the row softmax: tensor cores, one tile per row, 16-bit inputs only
    c = sel("bf16", 512, 512, 64, "nk", act="softmax")
    assert (c.kernel, c.bn, c.stages, c.variant, c.split_k) == ("tc", 512, 1, 1, 1)
    c = sel("bf16", 4, 200, 4096, "nk", act="softmax")     # small M: still the tile kernel
    assert (c.kernel, c.bn, c.stages, c.variant) == ("tc", 256, 3, 1)
    for kw in (dict(dtype="f32"), dict(N=513), dict(K=0), dict(residual=True)):
        args = dict(dtype="bf16", M=64, N=300, K=64)
        args.update({k: v for k, v in kw.items() if k in ("dtype", "N", "K")})
        with pytest.raises(g13.GemmError) as ei:
            sel(args["dtype"], args["M"], args["N"], args["K"], "nk", act="softmax",
                residual=kw.get("residual", False))
        assert ei.value.status == -2, kw



def test_dispatch_staging_follows_alignment(lib):
    # K = 3001 bf16: row stride 6002 B is not a multiple of 16 -> stage A (and B in NK)
    c = sel("bf16", 1000, 1000, 3001, "kn")
    assert (c.stage_a, c.stage_b) == (1, 0)
    c = sel("bf16", 1000, 1000, 3001, "nk")
    assert (c.stage_a, c.stage_b) == (1, 1)
    c = sel("bf16", 1000, 4097, 1000, "kn")
    assert (c.stage_a, c.stage_b) == (0, 1)
    c = sel("bf16", 1000, 1000, 6144, "kn")
    assert (c.stage_a, c.stage_b) == (0, 0)
    c = sel("f32", 3000, 3000, 302)     # 302*4 B rows: not 16-B aligned
    assert (c.kernel, c.stage_a, c.stage_b) == ("ffma", 1, 0)
    c = sel("f32", 300, 300, 302)       # small: 32 x 32 tiles from plain loads, no staging
    assert (c.kernel, c.variant, c.stage_a, c.stage_b) == ("ffma", 2, 0, 0)


def test_dispatch_bn_by_waves(lib):
    # 4096 x 1024 bf16 on 152 SMs: 32 x 4 = 128 tiles of 256 (one wave) vs 256 tiles of 128 (2 waves)
    assert sel("bf16", 4096, 1024, 4096, "nk").bn == 256
    # 512 x 512 x 96 heads: 384 tiles of 256 (3 waves) vs 768 of 128 (6 waves): same time, 256 wins
    assert sel("bf16", 512, 512, 64, "nk", batch=96, stride_a=512 * 64, stride_b=512 * 64,
               stride_c=512 * 512).bn == 256
    # 128 x 384: one tile of 256 + a half-empty one vs three tiles of 128 -> both one wave; 256 x2
    # waves equal, ratio decides
    c = sel("bf16", 128, 384, 4096, "nk", sms=2)
    assert c.bn in (128, 256)


def test_select_config_does_not_touch_cache(lib):
    g13.gemm_cache_clear()
    sel("bf16", 1024, 1024, 1024)
    assert g13.gemm_cache_stats() == (0, 0, 0)
