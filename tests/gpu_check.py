"""Shared helpers of the GPU parity tests: run a Workload through the C ABI and
compare the result with the FP64 oracle.

Tolerance (the stated acceptance bound for this GEMM), per output element:
    |C - C_ref| <= 2e-4 * L_act * S + 1e-6 (+ one ulp of |C_ref| in the
    output type when C is stored as BF16 or FP16)
where S = sum_k |a_ik * b_kj| comes from the oracle and L_act = 1.13 for GELU
(its largest slope), 1 otherwise.

Row softmax p = softmax(t), t = alpha*A.B + bias: with every t_k off by at
most d = 2e-4 * |alpha| * max_k S_ik (the bound above on the row), p_j moves
by at most p_j * (exp(2d) - 1); FP32 evaluation (the fast exponential, at
most ~6e-6 relative on [-88, 0]; four partial sums of up to 128 terms; one
product by 1/sum) adds at most 4e-5 * p_j; so
    |p - p_ref| <= p_ref * (expm1(2d) + 4e-5) + 1e-7 (+ one output ulp).

Output buffers carry guard bands: C lives inside a larger allocation filled
with NaN, and every element outside the M x N window must still be NaN after
the run (catches stores past tile edges).
"""
from __future__ import annotations

import numpy as np
import torch

import dense_gemm_13_gb300 as g13
import oracle
from dense_gemm_13_gb300.inputs import Workload, host_view

TORCH_OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
L_ACT = {"none": 1.0, "relu": 1.0, "gelu": 1.13}


def ulp(x: np.ndarray, out_dtype: str) -> np.ndarray:
    """One unit in the last place of |x| in the output format (0 for f32: not added)."""
    if out_dtype == "f32":
        return np.zeros_like(x)
    p, emin = (8, -126) if out_dtype == "bf16" else (11, -14)
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, emin)
    return np.where(ax > 0, 2.0 ** (e - (p - 1)), 2.0 ** (emin - (p - 1)))


def tolerance(sabs: np.ndarray, cref: np.ndarray, w: Workload) -> np.ndarray:
    if w.act == "softmax":      # sabs must hold whole rows
        d = 2e-4 * abs(w.alpha) * np.max(sabs, axis=-1, keepdims=True)
        return cref * (np.expm1(2 * d) + 4e-5) + 1e-7 + ulp(cref, w.out_dtype)
    return 2e-4 * L_ACT[w.act] * sabs + 1e-6 + ulp(cref, w.out_dtype)


class Run:
    """One library run of a workload, keeping host copies for the oracle."""

    def __init__(self, w: Workload, tensors: dict | None = None, config: g13.Config | None = None,
                 seed: int = 0, guard: bool = True, a_offset: int = 0, b_offset: int = 0,
                 plan: g13.Plan | None = None, ldc_pad: int = 0, flags: int = 0):
        self.w = w
        self.t = tensors if tensors is not None else w.make(seed)
        dev = torch.device("cuda")
        A, B = self.t["A"], self.t["B"]
        # optional misaligned views: operand starts `offset` elements into a buffer
        self.dA = self._place(A, a_offset, dev)
        self.dB = self._place(B, b_offset, dev)
        self.dbias = self.t["bias"].to(dev) if self.t["bias"] is not None else None
        self.dR = self.t["R"].to(dev) if self.t["R"] is not None else None
        bt, M, N = w.batch, w.M, w.N
        odt = TORCH_OUT[w.out_dtype]
        # guard bands: one NaN row above and below, 8 NaN columns on the left and
        # at least 8 on the right; C's start and row stride stay 16-byte aligned
        # (the TMA-store epilogue) unless ldc_pad makes the row stride odd (the
        # per-thread fallback).
        self.g = 1 if guard else 0
        self.ldc = ((N + 7) // 8 * 8 + 16 if guard else max(N, 1)) + ldc_pad
        self.cbuf = torch.full((bt, M + 2 * self.g, self.ldc), float("nan"), dtype=odt, device=dev)
        self.C = self.cbuf[:, self.g:self.g + M, 8 * self.g:8 * self.g + N]
        lda = A.shape[-1] if A.shape[-1] > 0 else 1
        ldb = B.shape[-1] if B.shape[-1] > 0 else 1
        ep = g13.Epilogue(b_layout=w.b_layout, out_dtype=w.out_dtype, bias=w.bias, act=w.act,
                          residual=w.residual, beta=w.beta,
                          ldr=(N if w.residual else 0) or 0, batch=bt,
                          stride_a=(w.M * w.K if (bt > 1 and A.dim() == 3) else 0),
                          stride_b=(B.shape[-1] * B.shape[-2] if (bt > 1 and B.dim() == 3) else 0),
                          stride_c=self.cbuf.shape[-1] * self.cbuf.shape[-2] if bt > 1 else 0,
                          stride_r=(M * N if (bt > 1 and w.residual) else 0), flags=flags)
        if w.residual and N == 0:
            ep.ldr = 1
        self.plan = plan or g13.gemm_plan(w.dtype, M, N, w.K, lda, ldb, self.ldc, ep, config)
        self.info = self.plan.info()

    @staticmethod
    def _place(t: torch.Tensor, offset: int, dev):
        if offset == 0:
            return t.to(dev)
        flat = torch.zeros(t.numel() + offset + 64, dtype=t.dtype, device=dev)
        flat[offset:offset + t.numel()] = t.reshape(-1).to(dev)
        return flat[offset:offset + t.numel()].view(t.shape)

    def run(self, alpha: float | None = None):
        a = self.w.alpha if alpha is None else alpha
        g13.gemm_run(self.plan, self.dA.data_ptr(), self.dB.data_ptr(), self.C.data_ptr(),
                     self.dbias, self.dR, a)
        return self

    def result(self) -> np.ndarray:
        torch.cuda.synchronize()
        st = g13.gemm_plan_status(self.plan)
        assert st == 0, f"device status {g13.STATUS.get(st, st)}"
        return self.C.float().cpu().double().numpy()

    def guard_ok(self) -> bool:
        torch.cuda.synchronize()
        mask = torch.ones(self.cbuf.shape, dtype=torch.bool, device=self.cbuf.device)
        g = self.g
        mask[:, g:g + self.w.M, 8 * g:8 * g + self.w.N] = False
        return bool(torch.isnan(self.cbuf[mask].float()).all().item())

    # ------------------------------------------------------------ oracle
    def oracle(self, rows=None, cols=None, threads=0):
        w, t = self.w, self.t
        return oracle.gemm(host_view(t["A"]), host_view(t["B"]), b_layout=w.b_layout, dtype=w.dtype,
                           alpha=w.alpha, bias=None if t["bias"] is None else t["bias"].numpy(),
                           act=w.act, R=None if t["R"] is None else t["R"].numpy(), beta=w.beta,
                           out_dtype=w.out_dtype, rows=rows, cols=cols, threads=threads)

    def check(self, C: np.ndarray, rows=None, cols=None, label=""):
        """Element-wise comparison on the rows x cols cross product (None = all)."""
        assert cols is None or self.w.act != "softmax", "the softmax tolerance needs whole rows"
        _, cref, sabs = self.oracle(rows, cols)
        if C.ndim == 2:
            C = C[None]
        if cref.ndim == 2:
            cref, sabs = cref[None], sabs[None]
        got = C
        if rows is not None:
            got = got[:, rows]
        if cols is not None:
            got = got[:, :, cols]
        tol = tolerance(sabs, cref, self.w)
        err = np.abs(got - cref)
        bad = ~(err <= tol)
        if bad.any():
            idx = np.argwhere(bad)
            b, i, j = idx[0]
            ratio = np.nanmax(np.where(tol > 0, err / tol, np.inf))
            raise AssertionError(
                f"{self.w.name}{label}: {bad.sum()} / {bad.size} outside tolerance; worst err/tol "
                f"{ratio:.3g}; first at batch {b} row {(rows[i] if rows is not None else i)} col "
                f"{(cols[j] if cols is not None else j)}: got {got[b, i, j]!r} want {cref[b, i, j]!r} "
                f"tol {tol[b, i, j]:.3g} (config {self.info['config']})")
        return float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0

    def freivalds(self, C: np.ndarray, trials: int = 2, seed: int = 99):
        """Whole-matrix check for linear epilogues: |C x - v| <= sum_j |x_j| tol_ij.

        This catches NaNs, Infs and gross errors anywhere in C, not a wrong
        tile: at large K the bound on a row sum is far wider than what one
        128 x 256 tile of wrong values moves it by.  Tile coverage comes from
        the element-wise checks on `tile_indices` rows and columns."""
        w, t = self.w, self.t
        assert w.act == "none"
        rng = np.random.default_rng(seed)
        Cb = C if C.ndim == 3 else C[None]
        for _ in range(trials):
            x = rng.choice([-1.0, 1.0], w.N)
            v, wv = oracle.freivalds(host_view(t["A"]), host_view(t["B"]), x, b_layout=w.b_layout,
                                     dtype=w.dtype, alpha=w.alpha,
                                     bias=None if t["bias"] is None else t["bias"].numpy(),
                                     R=None if t["R"] is None else t["R"].numpy(), beta=w.beta)
            v = v if v.ndim == 2 else v[None]
            wv = wv if wv.ndim == 2 else wv[None]
            cx = Cb @ x
            bound = 2e-4 * wv + w.N * 1e-6 + np.abs(Cb) @ np.abs(x) * 2.0 ** -24 + 1e-9
            err = np.abs(cx - v)
            assert np.all(err <= bound), (
                f"{w.name}: Freivalds check failed, worst err/bound {np.max(err / bound):.3g}")


def boundary_indices(n: int, tiles=(64, 128, 256), extra: int = 6, seed: int = 5) -> np.ndarray:
    """Tile-edge indices (0, 1, t-1, t, t+1 for each tile size, n-2, n-1) plus random ones."""
    s = {0, 1, n - 1, n - 2}
    for t in tiles:
        for base in (t, 2 * t, (n // t) * t):
            s.update({base - 1, base, base + 1})
    rng = np.random.default_rng(seed + n)
    s.update(int(v) for v in rng.integers(0, max(n, 1), extra))
    return np.array(sorted(v for v in s if 0 <= v < n), dtype=np.int64)


def tile_indices(n: int, block: int = 128, seed: int = 7) -> np.ndarray:
    """The tile-edge indices of `boundary_indices` plus one index at a random
    offset inside every `block`-wide block of [0, n).

    Checking every column of these rows (and every row of these columns)
    element by element reaches every output tile of any tiling whose tile
    sides are multiples of `block` (128 x 128, 128 x 256, 256 x 256 CTA-pair
    tiles, the raster-group wraps and the later persistent waves alike)."""
    s = set(int(v) for v in boundary_indices(n, extra=4, seed=seed))
    rng = np.random.default_rng(seed * 7919 + n)
    for b0 in range(0, n, block):
        s.add(b0 + int(rng.integers(0, min(block, n - b0))))
    return np.array(sorted(s), dtype=np.int64)
