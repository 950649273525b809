"""Thin Python binding of libgemm13.so (the C ABI declared in include/gemm13.h).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  PyTorch is used for device memory and the current stream; tensors
are passed as raw device pointers.  If the shared object is missing or fails
to load, every call raises -- there is no fallback.

    import dense_gemm_13_gb300 as g13
    plan = g13.gemm_plan("bf16", M, N, K, lda, ldb, ldc, g13.Epilogue(b_layout="nk"))
    g13.gemm_run(plan, A, B, C, alpha=1.0)       # torch CUDA tensors
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["Epilogue", "Config", "Plan", "GemmError", "gemm_plan", "gemm_run", "gemm_plan_status",
           "gemm_plan_info", "gemm_select_config", "gemm_cache_stats", "gemm_cache_clear",
           "gemm_strerror", "gemm_version", "gemm_run_noalloc", "lib", "load", "matmul", "DTYPES", "ACTS", "LAYOUTS",
           "KERNELS", "LIB_PATH"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgemm13.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
ACTS = {"none": 0, "gelu": 1, "relu": 2, "softmax": 3}
LAYOUTS = {"kn": 0, "nk": 1}
KERNELS = {"auto": 0, "tc": 1, "ffma": 2, "skinny": 3, "tf32x3": 4}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}
FLAG_FP32_TENSOR = 0x1         # FP32 inputs may run as 3xTF32 on the tensor cores
FLAG_TEST_STALL = 0x80000000
FLAG_TEST_STALL_PEER = 0x40000000   # test only: the second CTA withholds a tile

STATUS = {0: "GEMM_OK", -1: "GEMM_ERR_INVALID_ARG", -2: "GEMM_ERR_UNSUPPORTED",
          -3: "GEMM_ERR_MISALIGNED", -4: "GEMM_ERR_CUDA", -5: "GEMM_ERR_DEVICE_TIMEOUT",
          -6: "GEMM_ERR_BAD_PLAN", -7: "GEMM_ERR_NO_DEVICE", -8: "GEMM_ERR_OUT_OF_MEMORY",
          -9: "GEMM_ERR_SCRATCH_LIMIT"}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {name} ({_strerror(status)})" if what else name)


class _Epilogue(ctypes.Structure):
    _fields_ = [("b_layout", ctypes.c_int), ("out_dtype", ctypes.c_int), ("has_bias", ctypes.c_int),
                ("act", ctypes.c_int), ("has_residual", ctypes.c_int), ("beta", ctypes.c_float),
                ("ldr", ctypes.c_int64), ("batch", ctypes.c_int64), ("stride_a", ctypes.c_int64),
                ("stride_b", ctypes.c_int64), ("stride_c", ctypes.c_int64),
                ("stride_r", ctypes.c_int64), ("flags", ctypes.c_uint32),
                ("timeout_ms", ctypes.c_uint32)]


class _Config(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("bm", ctypes.c_int32), ("bn", ctypes.c_int32),
                ("bk", ctypes.c_int32), ("stages", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("raster_group", ctypes.c_int32), ("stage_a", ctypes.c_int32),
                ("stage_b", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("stream_k", ctypes.c_int32)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("config", _Config), ("workspace_bytes", ctypes.c_int64),
                ("num_sms", ctypes.c_int32), ("device", ctypes.c_int32),
                ("cache_hit", ctypes.c_int32), ("kernels_per_run", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libgemm13.so (built by __graft_entry__.build() / _build.build())."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -m dense_gemm_13_gb300._build`"
                               " (no fallback path exists)")
        L = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.gemm_epilogue_init.argtypes = [ctypes.POINTER(_Epilogue)]
        L.gemm_epilogue_init.restype = None
        L.gemm_plan.argtypes = [i32, i64, i64, i64, i64, i64, i64, ctypes.POINTER(_Epilogue),
                                ctypes.POINTER(vp)]
        L.gemm_plan.restype = i32
        L.gemm_plan_with_config.argtypes = [i32, i64, i64, i64, i64, i64, i64,
                                            ctypes.POINTER(_Epilogue), ctypes.POINTER(_Config),
                                            ctypes.POINTER(vp)]
        L.gemm_plan_with_config.restype = i32
        L.gemm_run.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp]
        L.gemm_run.restype = i32
        L.gemm_plan_status.argtypes = [vp]
        L.gemm_plan_status.restype = i32
        L.gemm_plan_info.argtypes = [vp, ctypes.POINTER(_PlanInfo)]
        L.gemm_plan_info.restype = i32
        L.gemm_plan_destroy.argtypes = [vp]
        L.gemm_plan_destroy.restype = None
        L.gemm_select_config.argtypes = [i32, i64, i64, i64, i64, i64, i64,
                                         ctypes.POINTER(_Epilogue), ctypes.c_int32,
                                         ctypes.POINTER(_Config)]
        L.gemm_select_config.restype = i32
        L.gemm_cache_stats.argtypes = [ctypes.POINTER(i64)] * 3
        L.gemm_cache_stats.restype = None
        L.gemm_cache_clear.argtypes = []
        L.gemm_cache_clear.restype = None
        L.gemm_strerror.argtypes = [i32]
        L.gemm_strerror.restype = ctypes.c_char_p
        L.gemm_version.argtypes = []
        L.gemm_version.restype = ctypes.c_char_p
        L.gemm_run_noalloc.argtypes = [i32, i64, i64, i64, vp, i64, vp, i64, vp, i64,
                                       ctypes.POINTER(_Epilogue), vp, vp, ctypes.c_float, vp]
        L.gemm_run_noalloc.restype = i32
        if path is None:
            _lib = L
        return L


def lib() -> ctypes.CDLL:
    return load()


def _strerror(status: int) -> str:
    try:
        return lib().gemm_strerror(status).decode()
    except Exception:
        return "?"


def gemm_strerror(status: int) -> str:
    return lib().gemm_strerror(int(status)).decode()


def gemm_version() -> str:
    return lib().gemm_version().decode()


class Epilogue:
    """Python mirror of gemm_epilogue_t (defaults as in gemm_epilogue_init)."""

    def __init__(self, b_layout="kn", out_dtype="f32", bias=False, act="none", residual=False,
                 beta=1.0, ldr=0, batch=1, stride_a=0, stride_b=0, stride_c=0, stride_r=0,
                 flags=0, timeout_ms=0):
        self.b_layout, self.out_dtype, self.bias, self.act = b_layout, out_dtype, bias, act
        self.residual, self.beta, self.ldr, self.batch = residual, beta, ldr, batch
        self.stride_a, self.stride_b, self.stride_c, self.stride_r = stride_a, stride_b, stride_c, stride_r
        self.flags, self.timeout_ms = flags, timeout_ms

    def _c(self) -> _Epilogue:
        e = _Epilogue()
        lib().gemm_epilogue_init(ctypes.byref(e))
        e.b_layout = LAYOUTS[self.b_layout]
        e.out_dtype = DTYPES[self.out_dtype]
        e.has_bias = int(bool(self.bias))
        e.act = ACTS[self.act]
        e.has_residual = int(bool(self.residual))
        e.beta = float(self.beta)
        e.ldr, e.batch = int(self.ldr), int(self.batch)
        e.stride_a, e.stride_b = int(self.stride_a), int(self.stride_b)
        e.stride_c, e.stride_r = int(self.stride_c), int(self.stride_r)
        e.flags, e.timeout_ms = int(self.flags), int(self.timeout_ms)
        return e


class Config:
    """Python mirror of gemm_config_t."""

    def __init__(self, kernel="auto", bm=0, bn=0, bk=0, stages=0, split_k=1, raster_group=0,
                 stage_a=0, stage_b=0, num_ctas=0, variant=0, stream_k=0):
        self.kernel, self.bm, self.bn, self.bk, self.stages = kernel, bm, bn, bk, stages
        self.split_k, self.raster_group, self.stage_a, self.stage_b = split_k, raster_group, stage_a, stage_b
        self.num_ctas, self.variant, self.stream_k = num_ctas, variant, stream_k

    def _c(self) -> _Config:
        c = _Config()
        c.kernel = KERNELS[self.kernel]
        c.bm, c.bn, c.bk, c.stages = self.bm, self.bn, self.bk, self.stages
        c.split_k, c.raster_group = self.split_k, self.raster_group
        c.stage_a, c.stage_b, c.num_ctas = self.stage_a, self.stage_b, self.num_ctas
        c.variant, c.stream_k = self.variant, self.stream_k
        return c

    @staticmethod
    def _from(c: _Config) -> "Config":
        return Config(KERNEL_NAMES.get(c.kernel, str(c.kernel)), c.bm, c.bn, c.bk, c.stages,
                      c.split_k, c.raster_group, c.stage_a, c.stage_b, c.num_ctas, c.variant,
                      c.stream_k)

    def as_dict(self) -> dict:
        return dict(kernel=self.kernel, bm=self.bm, bn=self.bn, bk=self.bk, stages=self.stages,
                    split_k=self.split_k, raster_group=self.raster_group, stage_a=self.stage_a,
                    stage_b=self.stage_b, num_ctas=self.num_ctas, variant=self.variant,
                    stream_k=self.stream_k)

    def __repr__(self):
        return f"Config({self.as_dict()})"


class Plan:
    """Owns a gemm_plan_t; destroyed with the object (or explicitly)."""

    def __init__(self, handle: int, dtype: str, M: int, N: int, K: int, epilogue: Epilogue):
        self.handle = handle
        self.dtype, self.M, self.N, self.K, self.epilogue = dtype, M, N, K, epilogue

    def destroy(self):
        if self.handle:
            lib().gemm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def run(self, A, B, C, bias=None, residual=None, alpha=1.0, stream=None):
        return gemm_run(self, A, B, C, bias, residual, alpha, stream)

    def info(self) -> dict:
        return gemm_plan_info(self)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def gemm_plan(dtype: str, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
              epilogue: Epilogue | None = None, config: Config | None = None) -> Plan:
    """gemm_plan / gemm_plan_with_config; raises GemmError on a non-OK status."""
    ep = epilogue or Epilogue()
    h = ctypes.c_void_p()
    ce = ep._c()
    if config is None:
        rc = lib().gemm_plan(DTYPES[dtype], M, N, K, lda, ldb, ldc, ctypes.byref(ce), ctypes.byref(h))
    else:
        cc = config._c()
        rc = lib().gemm_plan_with_config(DTYPES[dtype], M, N, K, lda, ldb, ldc, ctypes.byref(ce),
                                         ctypes.byref(cc), ctypes.byref(h))
    if rc != 0:
        raise GemmError(rc, "gemm_plan")
    return Plan(h.value, dtype, M, N, K, ep)


def gemm_run(plan: Plan, A, B, C, bias=None, residual=None, alpha: float = 1.0, stream=None) -> int:
    """Enqueue one GEMM on `stream` (default: torch's current stream); raises on error."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    rc = lib().gemm_run(plan.handle, _ptr(A), _ptr(B), _ptr(C), _ptr(bias), _ptr(residual),
                        float(alpha), stream)
    if rc != 0:
        raise GemmError(rc, "gemm_run")
    return rc


def gemm_plan_status(plan: Plan) -> int:
    """Synchronise and return the plan's sticky device status (0 or a negative code)."""
    return int(lib().gemm_plan_status(plan.handle))


def gemm_plan_info(plan: Plan) -> dict:
    info = _PlanInfo()
    rc = lib().gemm_plan_info(plan.handle, ctypes.byref(info))
    if rc != 0:
        raise GemmError(rc, "gemm_plan_info")
    return dict(config=Config._from(info.config), workspace_bytes=info.workspace_bytes,
                num_sms=info.num_sms, device=info.device, cache_hit=bool(info.cache_hit),
                kernels_per_run=info.kernels_per_run)


def gemm_select_config(dtype: str, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                       epilogue: Epilogue | None = None, num_sms: int = 152) -> Config:
    """Host-only dispatcher query (no GPU needed)."""
    ep = (epilogue or Epilogue())._c()
    c = _Config()
    rc = lib().gemm_select_config(DTYPES[dtype], M, N, K, lda, ldb, ldc, ctypes.byref(ep), num_sms,
                                  ctypes.byref(c))
    if rc != 0:
        raise GemmError(rc, "gemm_select_config")
    return Config._from(c)


def gemm_cache_stats() -> tuple[int, int, int]:
    e, h, m = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    lib().gemm_cache_stats(ctypes.byref(e), ctypes.byref(h), ctypes.byref(m))
    return e.value, h.value, m.value


def gemm_cache_clear() -> None:
    lib().gemm_cache_clear()


def gemm_run_noalloc(dtype: str, M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int,
                     epilogue: Epilogue | None = None, bias=None, residual=None,
                     alpha: float = 1.0, stream=None) -> int:
    """gemm_run_noalloc: one GEMM without any allocation (fixed in-library scratch).

    For callers that cannot allocate device memory where they run the GEMM;
    see include/gemm13.h for the scratch limit and the sharing rules.
    """
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    ce = (epilogue or Epilogue())._c()
    rc = lib().gemm_run_noalloc(DTYPES[dtype], M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                                ctypes.byref(ce), _ptr(bias), _ptr(residual), float(alpha), stream)
    if rc != 0:
        raise GemmError(rc, "gemm_run_noalloc")
    return rc


_plans: dict = {}


def matmul(A, B, *, b_layout="kn", alpha=1.0, bias=None, act="none", residual=None, beta=1.0,
           out_dtype="f32", out=None):
    """C = cast(act(alpha*A@B + bias) + beta*residual) for 2-D or 3-D (batched) CUDA tensors.

    Plans are created once per (shape, dtype, strides, epilogue) and kept.
    """
    import torch
    tdt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
    dt = tdt[A.dtype]
    batched = A.dim() == 3
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1] if b_layout == "kn" else B.shape[-2]
    batch = A.shape[0] if batched else 1
    odt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    if out is None:
        out = torch.empty((batch, M, N) if batched else (M, N), dtype=odt, device=A.device)
    lda, ldb, ldc = A.stride(-2), B.stride(-2), out.stride(-2)
    ep = Epilogue(b_layout=b_layout, out_dtype=out_dtype, bias=bias is not None, act=act,
                  residual=residual is not None, beta=beta,
                  ldr=residual.stride(-2) if residual is not None else 0, batch=batch,
                  stride_a=A.stride(0) if batched else 0,
                  stride_b=B.stride(0) if (batched and B.dim() == 3) else 0,
                  stride_c=out.stride(0) if batched else 0,
                  stride_r=residual.stride(0) if (batched and residual is not None and residual.dim() == 3) else 0)
    key = (dt, M, N, K, lda, ldb, ldc, tuple(sorted(vars(ep).items())), A.device.index)
    pl = _plans.get(key)
    if pl is None:
        pl = gemm_plan(dt, M, N, K, lda, ldb, ldc, ep)
        _plans[key] = pl
    gemm_run(pl, A, B, out, bias, residual, alpha)
    return out
