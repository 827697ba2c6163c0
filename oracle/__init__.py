"""CPU fp64 oracle for the BF16 GEMM and the implicit-GEMM convolution.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline may import this package; the library under
``mbarrier_pipelined_tensor_gb300`` never does, and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain loops, fp64 accumulation, the
textbook definitions). This file loads it and states the acceptance rule.

Acceptance (the error bound the mainloop must meet for the fp32 accumulator
before any bf16 rounding): per element
``|gpu - ref| <= 1e-3 * abs + 1e-6`` where ``abs = sum |a*b|`` over the same
terms. For bf16 outputs, half a bf16 ulp of the true value is added:
``+ 2**-8 * |ref|`` (round to nearest even of an in-tolerance fp32 value).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation tests load a deliberately broken build.
        path = os.environ.get("ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_gemm.argtypes = [p, p, i64, i64, i64, i64, i64, p, i64, p, i64, p, p]
        lib.oracle_gemm.restype = None
        lib.oracle_conv.argtypes = [p, p] + [i64] * 9 + [p, i64, p, p]
        lib.oracle_conv.restype = None
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_threads())


def gemm(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, lda: int, ldb: int,
         rows=None, cols=None):
    """fp64 C = A.B (and sum |a.b|) for the given rows x cols of C.

    A: uint16 bf16 bits, >= M*lda elements, a(i,k) = A[i*lda+k].
    B: uint16 bf16 bits, >= N*ldb elements, b(k,j) = B[j*ldb+k].
    rows/cols: index arrays (None = all). Returns (ref, abs), each
    len(rows) x len(cols) float64.
    """
    A = np.ascontiguousarray(A, dtype=np.uint16).reshape(-1)
    B = np.ascontiguousarray(B, dtype=np.uint16).reshape(-1)
    assert A.size >= (M - 1) * lda + K if M > 0 and K > 0 else True
    assert B.size >= (N - 1) * ldb + K if N > 0 and K > 0 else True
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    if r is not None:
        assert r.size == 0 or (r.min() >= 0 and r.max() < M)
    if c is not None:
        assert c.size == 0 or (c.min() >= 0 and c.max() < N)
    ref = np.zeros((nr, nc), dtype=np.float64)
    ab = np.zeros((nr, nc), dtype=np.float64)
    if nr and nc:
        _load().oracle_gemm(_ptr(A), _ptr(B), M, N, K, lda, ldb,
                            _ptr(r), nr, _ptr(c), nc, _ptr(ref), _ptr(ab))
    return ref, ab


def conv_out_hw(H, W, R, S, stride, pad):
    return (H + 2 * pad - R) // stride + 1, (W + 2 * pad - S) // stride + 1


def conv(x: np.ndarray, w: np.ndarray, N, H, W, C, K, R, S, stride, pad, pixels=None):
    """fp64 forward convolution (cross-correlation, zero padding).

    x: uint16 NHWC, w: uint16 KRSC. pixels: linear output-pixel indices
    n*P*Q + p*Q + q (None = all). Returns (ref, abs), each len(pixels) x K.
    """
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    w = np.ascontiguousarray(w, dtype=np.uint16).reshape(-1)
    assert x.size == N * H * W * C and w.size == K * R * S * C
    P, Q = conv_out_hw(H, W, R, S, stride, pad)
    px = None if pixels is None else np.ascontiguousarray(pixels, dtype=np.int64)
    npx = N * P * Q if px is None else px.size
    if px is not None:
        assert px.size == 0 or (px.min() >= 0 and px.max() < N * P * Q)
    ref = np.zeros((npx, K), dtype=np.float64)
    ab = np.zeros((npx, K), dtype=np.float64)
    if npx and K:
        _load().oracle_conv(_ptr(x), _ptr(w), N, H, W, C, K, R, S, stride, pad,
                            _ptr(px), npx, _ptr(ref), _ptr(ab))
    return ref, ab


# ---------------------------------------------------------------------------
# Acceptance
# ---------------------------------------------------------------------------

def tolerance(ref: np.ndarray, ab: np.ndarray, out_bf16: bool) -> np.ndarray:
    tol = 1e-3 * ab + 1e-6
    if out_bf16:
        tol = tol + np.abs(ref) * 2.0 ** -8
    return tol


def check(got: np.ndarray, ref: np.ndarray, ab: np.ndarray, out_bf16: bool):
    """Returns (ok, worst_ratio, n_bad). worst_ratio = max |err| / tol."""
    got = np.asarray(got, dtype=np.float64)
    tol = tolerance(ref, ab, out_bf16)
    err = np.abs(got - ref)
    bad = ~(err <= tol)          # NaN counts as bad
    ratio = float(np.max(np.where(np.isfinite(err), err / tol, np.inf))) if err.size else 0.0
    return (not bad.any()), ratio, int(bad.sum())


def sample_rows(M: int, every: int = 32) -> np.ndarray:
    """Deterministic row sample: every ``every``-th row plus the last."""
    r = list(range(0, M, every))
    if M - 1 not in r:
        r.append(M - 1)
    return np.asarray(r, dtype=np.int64)
