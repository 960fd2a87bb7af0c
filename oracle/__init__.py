"""CPU oracle for C = alpha*A*B + beta*C on row-major float32 matrices.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The library
path (``dense_fp32_matrix_sm_gb300``) never does, and this package imports
nothing from it.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, fp64, one definition
written out; see that file's header for the passages it follows).  This
module only marshals numpy arrays into it, plus ``bruteforce_py``: an
independent pure-Python loop used to pin the C code on tiny inputs.

Every function here returns float64 results and never rounds them to fp32.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_f64 = ctypes.c_double
_fp = ctypes.POINTER(ctypes.c_float)
_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile sgemm_oracle.c into liboracle.so next to it (gcc, no GPU)."""
    from .build_oracle import build_oracle

    return build_oracle(force=force)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    lib.oracle_sgemm.restype = ctypes.c_int
    lib.oracle_sgemm.argtypes = [_i64, _i64, _i64, _f64, _fp, _i64, _fp, _i64, _f64, _fp, _i64,
                                 _dp, _dp, _i64, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]
    lib.oracle_sgemm_entries.restype = ctypes.c_int
    lib.oracle_sgemm_entries.argtypes = [_i64, _i64, _i64, _f64, _fp, _i64, _fp, _i64, _f64, _fp,
                                         _i64, _i64, _ip, _ip, _dp, _dp]
    lib.oracle_fp32_chain_entries.restype = ctypes.c_int
    lib.oracle_fp32_chain_entries.argtypes = [_i64, _i64, _i64, _fp, _i64, _fp, _i64, _i64, _ip,
                                              _ip, ctypes.POINTER(ctypes.c_float)]
    _lib = lib
    return lib


def _as_f32_2d(x, name):
    x = np.asarray(x)
    if x.dtype != np.float32:
        raise TypeError(f"{name} must be float32, got {x.dtype}")
    if x.ndim != 2:
        raise ValueError(f"{name} must be 2-D")
    if x.strides[1] != 4 or (x.shape[0] > 1 and x.strides[0] % 4 != 0):
        x = np.ascontiguousarray(x)
    return x


def _ld(x):
    return max(1, x.strides[0] // 4) if x.shape[0] > 1 else max(1, x.shape[1])


def _ptr(x, ctype=_fp):
    return x.ctypes.data_as(ctype) if x is not None else None


def _check(rc):
    if rc == -1:
        raise ValueError("oracle: invalid argument")
    if rc == -2:
        raise MemoryError("oracle: out of memory")
    if rc != 0:
        raise RuntimeError(f"oracle: status {rc}")


def sgemm_ref(A, B, C0=None, alpha: float = 1.0, beta: float = 0.0, threads: Optional[int] = None,
              with_bound: bool = True, count_fmas: bool = False):
    """Full fp64 C_ref (and S = |A||B| when with_bound) for row-major float32 A, B, C0.

    Returns (C_ref, S) or (C_ref, S, n_fma) when count_fmas.  S is None when
    with_bound is False.  beta == 0 never reads C0.
    """
    lib = _load()
    A = _as_f32_2d(A, "A")
    B = _as_f32_2d(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        C0 = _as_f32_2d(C0, "C0")
        if C0.shape != (M, N):
            raise ValueError("C0 shape mismatch")
        ldc = _ld(C0)
    else:
        C0 = None
        ldc = max(1, N)
    Cref = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_bound else None
    nfma = ctypes.c_uint64(0)
    if threads is None:
        threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    rc = lib.oracle_sgemm(M, N, K, float(alpha), _ptr(A), _ld(A) if K > 0 else 1, _ptr(B), _ld(B),
                          float(beta), _ptr(C0), ldc, _ptr(Cref, _dp), _ptr(S, _dp), max(1, N),
                          int(threads), ctypes.byref(nfma))
    _check(rc)
    if count_fmas:
        return Cref, S, int(nfma.value)
    return Cref, S


def sgemm_ref_entries(A, B, C0, alpha: float, beta: float, rows, cols) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 C_ref[rows[e], cols[e]] and S[rows[e], cols[e]], one dot product per entry."""
    lib = _load()
    A = _as_f32_2d(A, "A")
    B = _as_f32_2d(B, "B")
    M, K = A.shape
    N = B.shape[1]
    if beta != 0.0:
        C0 = _as_f32_2d(C0, "C0")
        ldc = _ld(C0)
    else:
        C0 = None
        ldc = max(1, N)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    if cols.size != n:
        raise ValueError("rows and cols differ in length")
    cref = np.empty(n, dtype=np.float64)
    s = np.empty(n, dtype=np.float64)
    rc = lib.oracle_sgemm_entries(M, N, K, float(alpha), _ptr(A), _ld(A) if K > 0 else 1, _ptr(B),
                                  _ld(B), float(beta), _ptr(C0), ldc, n, _ptr(rows, _ip),
                                  _ptr(cols, _ip), _ptr(cref, _dp), _ptr(s, _dp))
    _check(rc)
    return cref, s


def fp32_chain_entries(A, B, rows, cols) -> np.ndarray:
    """float32 fmaf chain over ascending k for the requested entries (a bitwise diagnostic)."""
    lib = _load()
    A = _as_f32_2d(A, "A")
    B = _as_f32_2d(B, "B")
    M, K = A.shape
    N = B.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(rows.size, dtype=np.float32)
    rc = lib.oracle_fp32_chain_entries(M, N, K, _ptr(A), _ld(A) if K > 0 else 1, _ptr(B), _ld(B),
                                       rows.size, _ptr(rows, _ip), _ptr(cols, _ip),
                                       out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    _check(rc)
    return out


def bruteforce_py(A, B, C0, alpha: float, beta: float):
    """Pure-Python j - i - p triple loop in fp64 (tiny inputs only).

    Independent of the C code: different loop order, Python floats (IEEE
    double), written straight from the definition of one output element.
    Returns (C_ref, S) as nested lists.
    """
    M, K = len(A), (len(A[0]) if len(A) else 0)
    N = len(B[0]) if len(B) else (len(C0[0]) if C0 is not None and len(C0) else 0)
    C = [[0.0] * N for _ in range(M)]
    S = [[0.0] * N for _ in range(M)]
    for j in range(N):
        for i in range(M):
            dot = 0.0
            sab = 0.0
            for p in range(K):
                a = float(A[i][p])
                b = float(B[p][j])
                dot += a * b
                sab += abs(a) * abs(b)
            c = alpha * dot if (K > 0 and alpha != 0.0) else 0.0
            if beta != 0.0:
                c += beta * float(C0[i][j])
            C[i][j] = c
            S[i][j] = sab
    return C, S


def acceptance_bound(K: int, S):
    """The elementwise parity bound |C - C_ref| <= 4*K*2^-24*S + 1e-6."""
    return 4.0 * K * 2.0 ** -24 * np.asarray(S, dtype=np.float64) + 1e-6
