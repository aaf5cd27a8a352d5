"""The CPU oracle for the pipelined tiled GEMM -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never loads it; the two
share no code.  ``oracle.c`` holds every computation (fp64 triple loop, exact
fp16/bf16 decoders, nearest-even rounding, the pages' shared-memory bound);
this module only compiles it with gcc and marshals numpy arrays through
ctypes.  Each function's citation is in ``oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1
_DT = {"f16": F16, "bf16": BF16}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-ffp-contract=off"]
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB points the tests at a deliberately broken copy of the
            # oracle (the mutation test); otherwise the oracle is built here.
            path = os.environ.get("ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            i64, p = ctypes.c_int64, ctypes.c_void_p
            L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f64.restype = ctypes.c_double
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_f64_to_f16.argtypes = [ctypes.c_double]
            L.oracle_f64_to_f16.restype = ctypes.c_uint16
            L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            L.oracle_f64_to_bf16.restype = ctypes.c_uint16
            L.oracle_decode.argtypes = [p, p, i64, ctypes.c_int]
            L.oracle_round.argtypes = [p, p, i64, ctypes.c_int]
            L.oracle_gemm.argtypes = [i64, i64, i64, p, p, ctypes.c_int, p, p]
            L.oracle_gemm.restype = ctypes.c_int
            L.oracle_gemm_entries.argtypes = [i64, i64, i64, p, p, ctypes.c_int, p, p, i64, p, p]
            L.oracle_gemm_entries.restype = ctypes.c_int
            L.oracle_gemm_rows.argtypes = [i64, i64, i64, p, p, ctypes.c_int, i64, i64, p]
            L.oracle_gemm_rows.restype = ctypes.c_int
            L.oracle_gemm_decoded_rows.argtypes = [i64, i64, i64, p, p, i64, i64, p]
            L.oracle_gemm_decoded_rows.restype = ctypes.c_int
            L.oracle_smem_bound.argtypes = [i64] * 5
            L.oracle_smem_bound.restype = i64
            L.oracle_max_stages.argtypes = [i64] * 5
            L.oracle_max_stages.restype = i64
            L.oracle_flops.argtypes = [i64] * 3
            L.oracle_flops.restype = ctypes.c_double
            L.oracle_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("operands must be uint16 bit patterns")
    return a


def decode(bits, dtype: str) -> np.ndarray:
    """Exact float64 values of 16-bit patterns of ``dtype``."""
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_decode(_ptr(b), _ptr(out), b.size, _DT[dtype])
    return out


def round_to(values, dtype: str) -> np.ndarray:
    """Nearest-even rounding of float64 values to ``dtype``; uint16 bits."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_round(_ptr(v), _ptr(out), v.size, _DT[dtype])
    return out


def gemm(A, B, dtype: str, want_scale: bool = True):
    """``R = A . B^T`` and ``S = |A| . |B|^T`` (per product) in float64.

    ``A``: M x K and ``B``: N x K uint16 bit patterns of ``dtype``.
    """
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    R = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if want_scale else None
    rc = lib().oracle_gemm(M, N, K, _ptr(A), _ptr(B), _DT[dtype], _ptr(R),
                           _ptr(S) if S is not None else None)
    if rc != 0:
        raise RuntimeError("oracle_gemm failed")
    return (R, S) if want_scale else R


def gemm_entries(A, B, dtype: str, rows, cols):
    """Entries ``(rows[t], cols[t])`` of ``A . B^T`` and their scales."""
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N, _ = B.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    R = np.empty(n, dtype=np.float64)
    S = np.empty(n, dtype=np.float64)
    rc = lib().oracle_gemm_entries(M, N, K, _ptr(A), _ptr(B), _DT[dtype], _ptr(rows), _ptr(cols),
                                   n, _ptr(R), _ptr(S))
    if rc != 0:
        raise RuntimeError("oracle_gemm_entries failed")
    return R, S


def gemm_rows(A, B, dtype: str, row0: int, nrows: int) -> np.ndarray:
    """Rows ``[row0, row0 + nrows)`` of ``A . B^T`` in float64."""
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N, _ = B.shape
    R = np.empty((nrows, N), dtype=np.float64)
    rc = lib().oracle_gemm_rows(M, N, K, _ptr(A), _ptr(B), _DT[dtype], row0, nrows, _ptr(R))
    if rc != 0:
        raise RuntimeError("oracle_gemm_rows failed")
    return R


def gemm_decoded_rows(Ad, Bd, row0: int, nrows: int) -> np.ndarray:
    """Rows ``[row0, row0 + nrows)`` of ``Ad . Bd^T`` for float64 operands
    already produced by :func:`decode` (same sums, same order as :func:`gemm`)."""
    Ad = np.ascontiguousarray(Ad, dtype=np.float64)
    Bd = np.ascontiguousarray(Bd, dtype=np.float64)
    M, K = Ad.shape
    N, _ = Bd.shape
    R = np.empty((nrows, N), dtype=np.float64)
    rc = lib().oracle_gemm_decoded_rows(M, N, K, _ptr(Ad), _ptr(Bd), row0, nrows, _ptr(R))
    if rc != 0:
        raise RuntimeError("oracle_gemm_decoded_rows failed")
    return R


def smem_bound(block_M: int, block_N: int, block_K: int, num_stages: int, elem_bytes: int = 2) -> int:
    return int(lib().oracle_smem_bound(block_M, block_N, block_K, num_stages, elem_bytes))


def max_stages(block_M: int, block_N: int, block_K: int, budget: int, elem_bytes: int = 2) -> int:
    return int(lib().oracle_max_stages(block_M, block_N, block_K, elem_bytes, budget))


def flops(M: int, N: int, K: int) -> float:
    return float(lib().oracle_flops(M, N, K))


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def ulp(values, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` numbers at each value's magnitude (float64).

    IEEE 754: with p significand bits and minimum normal exponent emin, the
    spacing for |x| in [2^e, 2^(e+1)) is 2^(e - p + 1) when e >= emin; below
    2^emin (subnormals, and zero) it is the subnormal step 2^(emin - p + 1).
    """
    p, emin = {"f16": (11, -14), "bf16": (8, -126), "f32": (24, -126)}[dtype]
    a = np.abs(np.asarray(values, dtype=np.float64))
    _, e = np.frexp(a)  # a = f * 2^e with f in [0.5, 1): |x| lies in [2^(e-1), 2^e)
    e = np.where(a == 0, emin, np.maximum(e - 1, emin))
    return np.ldexp(1.0, e - (p - 1))


def check(C, R, S, out_dtype: str):
    """Elementwise acceptance against the oracle.

    fp32 output: ``|C - R| <= 1e-4 * S + 1e-5``.  16-bit output adds one ulp
    of the output format at ``R``.  Every output must also meet the pages'
    ``rtol = atol = 1e-2`` check.  Returns (ok, worst_ratio, index).
    """
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - R)
    bound = 1e-4 * S + 1e-5
    if out_dtype != "f32":
        bound = bound + ulp(R, out_dtype)
    pages = 1e-2 + 1e-2 * np.abs(R)
    ratio = np.maximum(err / bound, err / pages)
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    if ratio.size == 0:
        return True, 0.0, 0
    idx = int(np.argmax(ratio))
    return bool(ratio.flat[idx] <= 1.0), float(ratio.flat[idx]), idx
