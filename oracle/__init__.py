"""FP64 CPU oracle for C = epilogue(alpha * A @ B): test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The library never calls it; it shares
no code with the CUDA path.  The arithmetic lives in ``gemm_oracle.c`` (a plain
i/j/k triple loop accumulating in double; its header states the definition it
follows: the "DeepGEMM" page, sec. 1.2 / 3.4, and the "CUDA Tile ... GEMM"
page, sec. 2, 4.1 and 5.1).  This module only marshals numpy arrays into it.

Inputs are numpy arrays: float32 for FP32 problems, float16 for FP16, and
uint16 bit patterns for BF16 (numpy has no bfloat16).  The last dimension must
be contiguous; a leading third dimension is the batch.

Every function is pinned by ``tests/test_oracle_pins.py`` (closed forms,
exact integer brute force, identities, library special cases), and the
mutation test ``tests/test_oracle_mutants.py`` checks that planted mistakes in
the C source fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
ACTS = {"none": 0, "gelu": 1, "relu": 2, "softmax": 3}
LAYOUTS = {"kn": 0, "nk": 1}


def compile_oracle(src: str, out: str) -> str:
    """gcc -O2 -fopenmp: one shared object from one C file."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into liboracle.so next to it (if stale)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, _LIB)
    return _LIB


def _dtype_of(a: np.ndarray, dtype: str | None) -> str:
    if dtype is not None:
        return dtype
    if a.dtype == np.float32:
        return "f32"
    if a.dtype == np.float16:
        return "f16"
    if a.dtype == np.uint16:
        return "bf16"
    raise TypeError(f"unsupported oracle input dtype {a.dtype}")


def _mat(a: np.ndarray):
    """(pointer, ld, batch stride, batch) for a 2-D or 3-D array, in elements."""
    if a.ndim not in (2, 3):
        raise ValueError("operands must be 2-D or 3-D")
    it = a.itemsize
    if a.size == 0:
        return a.ctypes.data, max(a.shape[-1], 1), 0, (a.shape[0] if a.ndim == 3 else 1)
    if a.shape[-1] > 1 and a.strides[-1] != it:
        raise ValueError("last dimension must be contiguous")
    ld = a.strides[-2] // it if a.shape[-2] > 1 else a.shape[-1]
    if a.ndim == 3:
        return a.ctypes.data, ld, (a.strides[0] // it if a.shape[0] > 1 else 0), a.shape[0]
    return a.ctypes.data, ld, 0, 1


def _shape(A, B, b_layout):
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1] if b_layout == "kn" else B.shape[-2]
    KB = B.shape[-2] if b_layout == "kn" else B.shape[-1]
    if KB != K:
        raise ValueError(f"inner dimensions differ: A has K={K}, B has K={KB}")
    return M, N, K


class Oracle:
    """ctypes view of one compiled oracle shared object."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.oracle_gemm.restype = i32
        lib.oracle_gemm.argtypes = [i32, i64, i64, i64, i64,
                                    vp, i64, i64, vp, i64, i64, i32,
                                    dbl, vp, i32, vp, i64, i64, dbl, i32,
                                    vp, i64, vp, i64, vp, vp, vp, i32]
        lib.oracle_freivalds.restype = i32
        lib.oracle_freivalds.argtypes = [i32, i64, i64, i64, i64,
                                         vp, i64, i64, vp, i64, i64, i32,
                                         dbl, vp, vp, i64, i64, dbl,
                                         vp, vp, vp, vp, vp]
        lib.oracle_decode_f16.restype = dbl
        lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = dbl
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_round_to.restype = dbl
        lib.oracle_round_to.argtypes = [i32, dbl]
        lib.oracle_act.restype = dbl
        lib.oracle_act.argtypes = [i32, dbl]
        lib.oracle_max_threads.restype = i32
        lib.oracle_max_threads.argtypes = []
        self.lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def decode_f16(self, bits: int) -> float:
        return float(self.lib.oracle_decode_f16(bits))

    def decode_bf16(self, bits: int) -> float:
        return float(self.lib.oracle_decode_bf16(bits))

    def round_to(self, out_dtype: str, x: float) -> float:
        return float(self.lib.oracle_round_to(DTYPES[out_dtype], x))

    def act(self, name: str, y: float) -> float:
        return float(self.lib.oracle_act(ACTS[name], y))

    def gemm(self, A: np.ndarray, B: np.ndarray, *, b_layout: str = "kn",
             dtype: str | None = None, alpha: float = 1.0, bias: np.ndarray | None = None,
             act: str = "none", R: np.ndarray | None = None, beta: float = 1.0,
             out_dtype: str = "f32", rows=None, cols=None, threads: int = 0):
        """Reference outputs (y, c, sabs), each float64 of shape [batch?, rows, cols].

        y: epilogue value before output rounding; c: y rounded (RNE) to
        out_dtype; sabs: sum_k |a_ik * bhat_kj|.  rows / cols optionally
        select a subset of output rows / columns.
        """
        dt = _dtype_of(A, dtype)
        M, N, K = _shape(A, B, b_layout)
        pa, lda, sa, ba = _mat(A)
        pb, ldb, sb, bb = _mat(B)
        batch = max(ba, bb)
        if ba not in (1, batch) or bb not in (1, batch):
            raise ValueError("batch sizes differ")
        pr, ldr, sr = None, 0, 0
        if R is not None:
            R = np.asarray(R)
            if R.dtype != np.float32:
                raise TypeError("residual must be float32")
            pr, ldr, sr, br = _mat(R)
            if br not in (1, batch):
                raise ValueError("residual batch differs")
            if br == 1:
                sr = 0
        pbias = None
        if bias is not None:
            bias = np.ascontiguousarray(bias, dtype=np.float32)
            if bias.shape != (N,):
                raise ValueError("bias must have shape [N]")
            pbias = bias.ctypes.data
        rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        cols_a = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
        nr = M if rows_a is None else len(rows_a)
        nc = N if cols_a is None else len(cols_a)
        y = np.empty((batch, nr, nc), np.float64)
        c = np.empty((batch, nr, nc), np.float64)
        s = np.empty((batch, nr, nc), np.float64)
        rc = self.lib.oracle_gemm(
            DTYPES[dt], M, N, K, batch,
            pa, lda, sa if ba > 1 else 0, pb, ldb, sb if bb > 1 else 0,
            LAYOUTS[b_layout], float(alpha), pbias, ACTS[act],
            pr, ldr, sr, float(beta), DTYPES[out_dtype],
            None if rows_a is None else rows_a.ctypes.data, nr,
            None if cols_a is None else cols_a.ctypes.data, nc,
            y.ctypes.data, c.ctypes.data, s.ctypes.data, int(threads))
        if rc != 0:
            raise ValueError("oracle_gemm rejected its arguments")
        if A.ndim == 2 and B.ndim == 2:
            return y[0], c[0], s[0]
        return y, c, s

    def freivalds(self, A: np.ndarray, B: np.ndarray, x: np.ndarray, *, b_layout: str = "kn",
                  dtype: str | None = None, alpha: float = 1.0, bias=None, R=None,
                  beta: float = 1.0):
        """(v, w) of shape [batch?, M] for a linear epilogue (no activation).

        v = exact C @ x; w_i = sum_k |a_ik| * sum_j |bhat_kj| |x_j|, which
        equals sum_j |x_j| * S_ij.
        """
        dt = _dtype_of(A, dtype)
        M, N, K = _shape(A, B, b_layout)
        pa, lda, sa, ba = _mat(A)
        pb, ldb, sb, bb = _mat(B)
        batch = max(ba, bb)
        x = np.ascontiguousarray(x, dtype=np.float64)
        if x.shape != (N,):
            raise ValueError("x must have shape [N]")
        pr, ldr, sr = None, 0, 0
        if R is not None:
            R = np.asarray(R)
            pr, ldr, sr, br = _mat(R)
            if br == 1:
                sr = 0
        pbias = None
        if bias is not None:
            bias = np.ascontiguousarray(bias, dtype=np.float32)
            pbias = bias.ctypes.data
        u = np.empty(max(K, 1), np.float64)
        ua = np.empty(max(K, 1), np.float64)
        v = np.empty((batch, M), np.float64)
        w = np.empty((batch, M), np.float64)
        rc = self.lib.oracle_freivalds(
            DTYPES[dt], M, N, K, batch,
            pa, lda, sa if ba > 1 else 0, pb, ldb, sb if bb > 1 else 0,
            LAYOUTS[b_layout], float(alpha), pbias, pr, ldr, sr, float(beta),
            x.ctypes.data, u.ctypes.data, ua.ctypes.data, v.ctypes.data, w.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_freivalds rejected its arguments")
        if A.ndim == 2 and B.ndim == 2:
            return v[0], w[0]
        return v, w


_lock = threading.Lock()
_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from gemm_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gemm(*args, **kw):
    return default().gemm(*args, **kw)


def freivalds(*args, **kw):
    return default().freivalds(*args, **kw)


def max_threads() -> int:
    return default().max_threads()
