"""Pins for the FP64 oracle: checks against facts that do not come from the oracle.

Each `check_*` function takes an `oracle.Oracle` and raises AssertionError on
a mismatch.  They are run as CPU tests (test_oracle_pins.py) against the real
oracle and, in test_oracle_mutants.py, against copies of it with planted
mistakes, every one of which must fail at least one check.

What pins what:
  * IEEE decode of FP16 / BF16 bit patterns: exhaustive, against numpy's and
    torch's own conversions (a library routine as a special case).
  * RNE rounding to f32 / f16 / bf16: against numpy / torch conversions and
    hand-made ties.
  * The activations: standard-normal-table values (tests/golden).
  * The triple loop: exact integer brute force in Python ints; identity and
    permutation matrices; all-ones (every entry = K); the transpose identity
    (AB)^T = B^T A^T bit-for-bit; KN vs NK layouts; float64 numpy matmul.
  * The epilogue order: hand-derived scalar chains (tests/golden).
  * Sampling, batching and strides: against the full / unbatched result.
  * The Freivalds vectors: against C @ x and S @ |x| of the full result.
  * The row softmax: scipy's softmax of the float64 product (a library
    routine), the two-column closed form (the logistic function), rows
    summing to one, no overflow for large logits, invariance to a constant
    shift of the bias, and sampled / batched outputs against the full ones.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _as(dtype, x: np.ndarray) -> np.ndarray:
    """float64 values (exactly representable) -> the oracle's input form."""
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "f16":
        return x.astype(np.float16)
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def check_decode(o):
    bits = np.arange(65536, dtype=np.uint16)
    ref16 = bits.view(np.float16).astype(np.float64)
    got16 = np.array([o.decode_f16(int(b)) for b in bits])
    fin = np.isfinite(ref16)
    assert np.array_equal(got16[fin], ref16[fin]), "f16 decode"
    assert np.all(np.isinf(got16[np.isinf(ref16)])) and np.all(np.isnan(got16[np.isnan(ref16)]))
    refb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().double().numpy()
    gotb = np.array([o.decode_bf16(int(b)) for b in bits])
    fin = np.isfinite(refb)
    assert np.array_equal(gotb[fin], refb[fin]), "bf16 decode"
    # a few fixed patterns by hand
    assert o.decode_f16(0x3C00) == 1.0 and o.decode_f16(0xC000) == -2.0
    assert o.decode_f16(0x7BFF) == 65504.0 and o.decode_f16(0x0001) == 2.0 ** -24
    assert o.decode_f16(0x0400) == 2.0 ** -14 and o.decode_bf16(0x3F80) == 1.0
    assert o.decode_bf16(0xC0A0) == -5.0


def check_round(o):
    rng = np.random.default_rng(7)
    # f32: numpy float64 -> float32 is round-to-nearest-even
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, 2000),
                        rng.standard_normal(200) * 1e-42])
    got = np.array([o.round_to("f32", float(v)) for v in x])
    assert np.array_equal(got, x.astype(np.float32).astype(np.float64)), "f32 rounding"
    # f16: numpy float64 -> float16 (correctly rounded, RNE), incl. subnormals / overflow
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-8, 5, 2000),
                        [65519.0, 65520.0, -70000.0, 2.0 ** -25, 3 * 2.0 ** -26]])
    got = np.array([o.round_to("f16", float(v)) for v in x])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, ref), "f16 rounding"
    # bf16: torch float32 -> bfloat16 is RNE; inputs exactly representable in float32
    x = (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().double().numpy()
    got = np.array([o.round_to("bf16", float(v)) for v in x])
    assert np.array_equal(got, ref), "bf16 rounding"
    # hand-made ties: bf16 has 8 significant bits, ulp(1) = 2^-7
    assert o.round_to("bf16", 1 + 2.0 ** -8) == 1.0
    assert o.round_to("bf16", 1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert o.round_to("bf16", -(1 + 2.0 ** -8 + 2.0 ** -30)) == -(1 + 2.0 ** -7)
    maxbf = (2 - 2.0 ** -7) * 2.0 ** 127
    assert o.round_to("bf16", maxbf) == maxbf
    assert math.isinf(o.round_to("bf16", maxbf + 2.0 ** 119))     # tie to even -> 2^128 -> inf
    assert o.round_to("f16", 1 + 2.0 ** -11) == 1.0                 # f16: ulp(1) = 2^-10
    assert o.round_to("f16", 1 + 3 * 2.0 ** -11) == 1 + 2.0 ** -9


def check_act(o):
    g = _golden("epilogue_points.json")
    for p in g["gelu"]:
        assert abs(o.act("gelu", p["y"]) - p["gelu"]) <= 1e-15 * max(1.0, abs(p["y"])), p
    assert o.act("relu", -1.5) == 0.0 and o.act("relu", 2.5) == 2.5 and o.act("relu", 0.0) == 0.0
    assert o.act("none", -3.25) == -3.25


def _brute(a, b):
    """Exact integer C and S by Python int arithmetic (no floating point)."""
    M, K = a.shape
    N = b.shape[1]
    C = [[sum(int(a[i, k]) * int(b[k, j]) for k in range(K)) for j in range(N)] for i in range(M)]
    S = [[sum(abs(int(a[i, k]) * int(b[k, j])) for k in range(K)) for j in range(N)] for i in range(M)]
    return np.array(C, dtype=np.float64), np.array(S, dtype=np.float64)


def check_brute_force(o):
    rng = np.random.default_rng(11)
    for trial in range(60):
        M, N, K = (int(v) for v in rng.integers(1, 9, 3))
        a = rng.integers(-4, 5, (M, K))
        b = rng.integers(-4, 5, (K, N))
        C, S = _brute(a, b)
        for dt in ("f32", "f16", "bf16"):
            A = _as(dt, a.astype(np.float64))
            for lay in ("kn", "nk"):
                Bm = _as(dt, (b if lay == "kn" else b.T.copy()).astype(np.float64))
                y, c, s = o.gemm(A, Bm, b_layout=lay, dtype=dt)
                assert np.array_equal(c, C), (trial, dt, lay)
                assert np.array_equal(s, S), (trial, dt, lay)
                assert np.array_equal(y, C)


def check_identity_permutation(o):
    rng = np.random.default_rng(12)
    n, N = 37, 29
    Bv = _as("bf16", rng.standard_normal((n, N)))
    Bd = torch.from_numpy(Bv.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    perm = rng.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    _, c, _ = o.gemm(_as("bf16", P), Bv, dtype="bf16")
    assert np.array_equal(c, Bd[perm]), "P @ B must permute rows"
    A = _as("f32", rng.standard_normal((23, n)))
    _, c, _ = o.gemm(A, _as("f32", np.eye(n)))
    assert np.array_equal(c, A.astype(np.float64)), "A @ I == A"
    _, c, _ = o.gemm(A, _as("f32", P.T.copy()))
    assert np.array_equal(c, A.astype(np.float64)[:, perm]), "A @ P^T permutes columns"


def check_all_ones(o):
    for K in (1, 17, 127, 1000, 6144):
        for dt in ("f32", "bf16", "f16"):
            A = _as(dt, np.ones((3, K)))
            B = _as(dt, np.ones((K, 5)))
            _, c, s = o.gemm(A, B, dtype=dt)
            assert np.all(c == K) and np.all(s == K), (K, dt)
            _, c, _ = o.gemm(A, B, dtype=dt, out_dtype="bf16")
            assert np.all(c == o.round_to("bf16", K))


def check_transpose_identity(o):
    rng = np.random.default_rng(13)
    for dt in ("f32", "bf16", "f16"):
        a = rng.standard_normal((19, 33))
        b = rng.standard_normal((33, 11))
        A, B = _as(dt, a), _as(dt, b)
        _, c1, s1 = o.gemm(A, B, dtype=dt)
        _, c2, s2 = o.gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), dtype=dt)
        assert np.array_equal(c1.T, c2) and np.array_equal(s1.T, s2), dt
        # the same product with B handed over as [N,K]
        _, c3, _ = o.gemm(A, np.ascontiguousarray(B.T), b_layout="nk", dtype=dt)
        assert np.array_equal(c1, c3), dt


def check_numpy_matmul(o):
    rng = np.random.default_rng(14)
    for dt in ("f32", "bf16", "f16"):
        for (M, N, K) in ((31, 47, 129), (8, 300, 1000)):
            A, B = _as(dt, rng.standard_normal((M, K))), _as(dt, rng.standard_normal((K, N)))
            ad = torch.from_numpy(A.view(np.int16).copy()).view(torch.bfloat16).double().numpy() \
                if dt == "bf16" else A.astype(np.float64)
            bd = torch.from_numpy(B.view(np.int16).copy()).view(torch.bfloat16).double().numpy() \
                if dt == "bf16" else B.astype(np.float64)
            ref = ad @ bd
            sref = np.abs(ad) @ np.abs(bd)
            y, _, s = o.gemm(A, B, dtype=dt)
            # float64 summation-order differences only: each side is within
            # K * 2^-53 * S of the exact value
            assert np.all(np.abs(y - ref) <= 2 * K * 2.0 ** -53 * sref), dt
            assert np.all(np.abs(s - sref) <= 2 * K * 2.0 ** -53 * sref), dt


def check_epilogue_chain(o):
    g = _golden("epilogue_points.json")
    for p in g["scalar_chain"]:
        A = np.array([[p["a"]]], np.float32)
        B = np.array([[p["b"]]], np.float32)
        y, c, _ = o.gemm(A, B, alpha=p["alpha"], bias=np.array([p["bias"]], np.float32),
                         act=p["act"], R=np.array([[p["R"]]], np.float32), beta=p["beta"])
        assert abs(y[0, 0] - p["y"]) <= 1e-15 * abs(p["y"]), p
        assert c[0, 0] == np.float32(y[0, 0])
    # alpha = 0 leaves act(bias) + beta R; zero A gives GELU(bias)
    rng = np.random.default_rng(15)
    M, N, K = 6, 9, 13
    A = _as("bf16", rng.standard_normal((M, K)))
    B = _as("bf16", rng.standard_normal((K, N)))
    bias = rng.standard_normal(N).astype(np.float32)
    R = rng.standard_normal((M, N)).astype(np.float32)
    y, _, _ = o.gemm(A, B, dtype="bf16", alpha=0.0, bias=bias, act="relu", R=R, beta=-0.5)
    assert np.array_equal(y, np.maximum(bias.astype(np.float64), 0)[None, :] - 0.5 * R.astype(np.float64))
    y, _, _ = o.gemm(_as("bf16", np.zeros((M, K))), B, dtype="bf16", bias=bias, act="gelu")
    g1 = np.array([o.act("gelu", float(v)) for v in bias])
    assert np.array_equal(y, np.broadcast_to(g1, (M, N)))
    # bf16 output is the RNE rounding of y
    y, c, _ = o.gemm(A, B, dtype="bf16", bias=bias, act="gelu", out_dtype="bf16")
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    exact32 = y.astype(np.float32).astype(np.float64) == y
    assert np.array_equal(c[exact32], ref[exact32])
    assert np.all(np.abs(c - y) <= 2.0 ** -8 * np.abs(y))


def check_sampling_batching(o):
    rng = np.random.default_rng(16)
    bt, M, N, K = 3, 21, 18, 40
    A = _as("f16", rng.standard_normal((bt, M, K)))
    B = _as("f16", rng.standard_normal((bt, N, K)))
    R = rng.standard_normal((bt, M, N)).astype(np.float32)
    bias = rng.standard_normal(N).astype(np.float32)
    kw = dict(b_layout="nk", dtype="f16", alpha=0.125, bias=bias, R=R, beta=0.75, act="relu")
    y, c, s = o.gemm(A, B, **kw)
    for b in range(bt):
        kwb = dict(kw, R=R[b])
        yb, cb, sb = o.gemm(A[b], B[b], **kwb)
        assert np.array_equal(yb, y[b]) and np.array_equal(sb, s[b]), b
    rows, cols = [0, 5, 20, 5], [17, 0, 3]
    ys, cs, ss = o.gemm(A, B, rows=rows, cols=cols, **kw)
    assert np.array_equal(ys, y[:, rows][:, :, cols]) and np.array_equal(ss, s[:, rows][:, :, cols])
    # padded leading dimensions (views of wider arrays)
    Aw = _as("f32", rng.standard_normal((M, K + 7)))
    Bw = _as("f32", rng.standard_normal((K, N + 5)))
    Rw = rng.standard_normal((M, N + 3)).astype(np.float32)
    y1, _, _ = o.gemm(Aw[:, :K], Bw[:, :N], R=Rw[:, :N])
    y2, _, _ = o.gemm(np.ascontiguousarray(Aw[:, :K]), np.ascontiguousarray(Bw[:, :N]),
                      R=np.ascontiguousarray(Rw[:, :N]))
    assert np.array_equal(y1, y2)


def check_sabs(o):
    rng = np.random.default_rng(17)
    a = np.abs(rng.standard_normal((9, 30)))
    b = np.abs(rng.standard_normal((30, 12)))
    y, _, s = o.gemm(_as("f32", a), _as("f32", b))
    assert np.array_equal(y, s), "nonnegative inputs: S == C"
    y2, _, s2 = o.gemm(_as("f32", -a), _as("f32", b))
    assert np.array_equal(s2, s) and np.array_equal(y2, -y)


def check_freivalds(o):
    rng = np.random.default_rng(18)
    for lay in ("kn", "nk"):
        M, N, K = 25, 31, 57
        A = _as("bf16", rng.standard_normal((M, K)))
        B = _as("bf16", rng.standard_normal((K, N) if lay == "kn" else (N, K)))
        bias = rng.standard_normal(N).astype(np.float32)
        R = rng.standard_normal((M, N)).astype(np.float32)
        x = rng.choice([-1.0, 1.0], N)
        y, _, s = o.gemm(A, B, b_layout=lay, dtype="bf16", alpha=0.5, bias=bias, R=R, beta=1.5)
        v, w = o.freivalds(A, B, x, b_layout=lay, dtype="bf16", alpha=0.5, bias=bias, R=R, beta=1.5)
        assert np.allclose(v, y @ x, rtol=1e-12, atol=1e-9), lay
        assert np.allclose(w, s @ np.abs(x), rtol=1e-12, atol=0), lay


def check_softmax(o):
    from scipy.special import softmax
    rng = np.random.default_rng(21)
    # scipy's softmax of the float64 product, per-column bias, NK layout (Q.K^T)
    M, N, K = 7, 11, 16
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    bias = rng.standard_normal(N).astype(np.float32)
    t = 0.125 * (A.astype(np.float64) @ B.astype(np.float64).T) + bias.astype(np.float64)
    y, c, sabs = o.gemm(A, B, b_layout="nk", alpha=0.125, bias=bias, act="softmax")
    assert np.allclose(y, softmax(t, axis=1), rtol=1e-12, atol=0)
    assert np.all(np.abs(y.sum(axis=1) - 1.0) <= 1e-14)
    assert np.array_equal(c, y.astype(np.float32).astype(np.float64))
    assert np.allclose(sabs, np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T,
                       rtol=1e-14)
    # two columns: p0 = 1 / (1 + exp(t1 - t0)); B = I (KN) makes t = A
    A2 = np.array([[1.0, 2.0], [3.0, -1.0], [0.5, 0.5]], np.float32)
    y, _, _ = o.gemm(A2, np.eye(2, dtype=np.float32), act="softmax")
    p0 = 1.0 / (1.0 + np.exp(A2[:, 1].astype(np.float64) - A2[:, 0]))
    assert np.allclose(y[:, 0], p0, rtol=1e-15) and np.allclose(y[:, 1], 1.0 - p0, rtol=1e-14)
    # large logits (alpha = 1000): no overflow, one-hot at the row maximum
    Ai = rng.integers(-4, 5, (5, 8)).astype(np.float32)
    Bi = rng.integers(-4, 5, (8, 9)).astype(np.float32)
    y, _, _ = o.gemm(Ai, Bi, alpha=1000.0, act="softmax")
    prod = Ai.astype(np.float64) @ Bi.astype(np.float64)
    assert np.all(np.isfinite(y)) and np.all(np.abs(y.sum(axis=1) - 1.0) <= 1e-14)
    for i in range(5):
        top = np.flatnonzero(prod[i] == prod[i].max())
        assert np.allclose(y[i, top], 1.0 / len(top), rtol=1e-12)
    # a constant added to every bias entry leaves p unchanged (eighths: the shift is exact)
    bq = (rng.integers(-16, 17, N) / 8).astype(np.float32)
    y1, _, _ = o.gemm(A, B, b_layout="nk", alpha=0.125, bias=bq, act="softmax")
    y2, _, _ = o.gemm(A, B, b_layout="nk", alpha=0.125, bias=bq + np.float32(3.0), act="softmax")
    assert np.allclose(y1, y2, rtol=1e-13, atol=0)
    # sampled rows / columns still see the whole row; batches are independent
    rows, cols = np.array([6, 0, 3]), np.array([10, 2, 5, 4])
    ys, _, _ = o.gemm(A, B, b_layout="nk", alpha=0.125, bias=bq, act="softmax", rows=rows,
                      cols=cols)
    assert np.array_equal(ys, y1[np.ix_(rows, cols)])
    Ab = rng.standard_normal((3, M, K)).astype(np.float32)
    Bb = rng.standard_normal((3, N, K)).astype(np.float32)
    yb, _, _ = o.gemm(Ab, Bb, b_layout="nk", alpha=0.5, act="softmax", out_dtype="bf16")
    for b in range(3):
        yo, _, _ = o.gemm(Ab[b], Bb[b], b_layout="nk", alpha=0.5, act="softmax")
        assert np.array_equal(yb[b], yo)
    # the row softmax takes no residual
    try:
        o.gemm(A, B, b_layout="nk", act="softmax", R=np.zeros((M, N), np.float32))
    except Exception:
        pass
    else:
        raise AssertionError("softmax with a residual was accepted")


ALL_CHECKS = [check_decode, check_round, check_act, check_brute_force, check_identity_permutation,
              check_all_ones, check_transpose_identity, check_numpy_matmul, check_epilogue_chain,
              check_sampling_batching, check_sabs, check_freivalds, check_softmax]
