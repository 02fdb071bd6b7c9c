"""CPU oracle for the dense GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library in
``dense_gemm_engineering_gb300``) never imports it, and this package imports
nothing from the product: the two share no code.

The arithmetic lives in ``gemm_oracle.c`` (plain C, binary64 accumulation, one
round-to-nearest-even step to the 16-bit output type).  This module compiles
it with gcc on first use and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgemm_oracle.so")

F16, BF16 = 0, 1
B_NK, B_KN = 0, 1  # B stored N x K (D = A.Bt) or K x N (D = A.B)


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library at ``out``.

    Uses OpenMP when the compiler supports it, else one thread.
    ``-ffp-contract=off`` keeps every multiply and add a separate IEEE
    operation (the products are exact in binary64 either way).
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", src, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``oracle/_build/libgemm_oracle.so``."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _dt(dtype) -> int:
    if dtype in ("f16", "fp16", "float16", F16):
        return F16
    if dtype in ("bf16", "bfloat16", BF16):
        return BF16
    raise ValueError(f"unknown dtype {dtype!r}")


class Oracle:
    """ctypes wrapper around one compiled oracle library."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_gemm.argtypes = [u16p, u16p, i64, i64, i64, i64, i64, ctypes.c_int,
                                    ctypes.c_int, i64, i64, i64, i64, u16p, f64p, i64]
        lib.oracle_gemm.restype = None
        lib.oracle_to_double.argtypes = [ctypes.c_uint16, ctypes.c_int]
        lib.oracle_to_double.restype = ctypes.c_double
        lib.oracle_from_double.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.oracle_from_double.restype = ctypes.c_uint16
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_fp8_to_double.argtypes = [ctypes.c_uint8, ctypes.c_int]
        lib.oracle_fp8_to_double.restype = ctypes.c_double
        lib.oracle_gemm_fp8.argtypes = [u8p, u8p, i64, i64, i64, i64, i64, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_double, i64, i64, i64, i64,
                                        u16p, f64p, i64]
        lib.oracle_gemm_fp8.restype = None
        lib.oracle_ue8m0_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_ue8m0_to_double.restype = ctypes.c_double
        lib.oracle_gemm_mx.argtypes = [u8p, u8p, u8p, u8p, i64, i64, i64, i64, i64, i64, i64,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_double, i64, i64, i64,
                                       i64, u16p, f64p, i64]
        lib.oracle_gemm_mx.restype = None
        self._lib = lib
        self.path = so_path

    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        """Threads for later calls (the OpenMP runtime's setting; n >= 1)."""
        self._lib.oracle_set_num_threads(int(n))

    def to_double(self, bits, dtype) -> np.ndarray:
        """Exact binary64 value of each 16-bit pattern."""
        d = _dt(dtype)
        b = np.asarray(bits, dtype=np.uint16)
        return np.array([self._lib.oracle_to_double(int(x), d) for x in b.ravel()],
                        dtype=np.float64).reshape(b.shape)

    def from_double(self, x, dtype) -> np.ndarray:
        """Round binary64 values to 16-bit patterns (nearest, ties to even)."""
        d = _dt(dtype)
        a = np.asarray(x, dtype=np.float64)
        return np.array([self._lib.oracle_from_double(float(v), d) for v in a.ravel()],
                        dtype=np.uint16).reshape(a.shape)

    def gemm(self, A, B, *, layout: str = "abt", dtype="f16", rows=None, cols=None,
             want_f64: bool = False):
        """Oracle GEMM on 16-bit patterns.

        A: (M, K) uint16 patterns (any 2-D view with unit inner stride, so the
        row stride may exceed K).  B: (N, K) for ``layout="abt"`` (D = A.Bt)
        or (K, N) for ``layout="ab"`` (D = A.B).  ``rows``/``cols`` are
        (start, stop) ranges of D to compute (default: all of D).  Returns the
        uint16 patterns of D[rows, cols] and, with ``want_f64``, also the
        unrounded binary64 sums.
        """
        d = _dt(dtype)
        A = np.asarray(A)
        B = np.asarray(B)
        if A.dtype != np.uint16 or B.dtype != np.uint16:
            raise TypeError("oracle.gemm takes uint16 bit patterns")
        if A.ndim != 2 or B.ndim != 2:
            raise ValueError("operands must be 2-D")
        if A.size and A.strides[1] != 2:
            A = np.ascontiguousarray(A)
        if B.size and B.strides[1] != 2:
            B = np.ascontiguousarray(B)
        M, K = A.shape
        if layout == "abt":
            N, Kb = B.shape
            bl = B_NK
        elif layout == "ab":
            Kb, N = B.shape
            bl = B_KN
        else:
            raise ValueError(f"unknown layout {layout!r}")
        if Kb != K:
            raise ValueError(f"K mismatch: {K} vs {Kb}")
        i0, i1 = rows if rows is not None else (0, M)
        j0, j1 = cols if cols is not None else (0, N)
        if not (0 <= i0 <= i1 <= M and 0 <= j0 <= j1 <= N):
            raise ValueError("rows/cols out of range")
        lda = A.strides[0] // 2 if A.shape[0] > 1 else max(A.shape[1], 1)
        ldb = B.strides[0] // 2 if B.shape[0] > 1 else max(B.shape[1], 1)
        out16 = np.zeros((i1 - i0, j1 - j0), dtype=np.uint16)
        out64 = np.zeros((i1 - i0, j1 - j0), dtype=np.float64) if want_f64 else None
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        a_ptr = A.ctypes.data_as(u16p) if A.size else None
        b_ptr = B.ctypes.data_as(u16p) if B.size else None
        if out16.size:
            self._lib.oracle_gemm(a_ptr, b_ptr, M, N, K, lda, ldb, bl, d, i0, i1, j0, j1,
                                  out16.ctypes.data_as(u16p),
                                  out64.ctypes.data_as(f64p) if want_f64 else None, j1 - j0)
        return (out16, out64) if want_f64 else out16


def _fp8(fmt) -> int:
    if fmt in ("e4m3", 0):
        return 0
    if fmt in ("e5m2", 1):
        return 1
    raise ValueError(f"unknown FP8 format {fmt!r}")


def _fp8_methods():
    def fp8_to_double(self, bits, fmt) -> np.ndarray:
        """Exact binary64 value of each FP8 pattern (E4M3 or E5M2)."""
        f = _fp8(fmt)
        b = np.asarray(bits, dtype=np.uint8)
        return np.array([self._lib.oracle_fp8_to_double(int(v), f) for v in b.ravel()],
                        dtype=np.float64).reshape(b.shape)

    def gemm_fp8(self, A, B, *, fmt="e4m3", out_dtype="bf16", alpha=1.0, rows=None, cols=None,
                 want_f64: bool = False):
        """Oracle FP8 GEMM: D = round(alpha * A . Bt), A (M, K) and B (N, K) uint8
        FP8 patterns (K-major, unit inner stride), D as 16-bit patterns of
        ``out_dtype``.  ``alpha`` is used at its binary32 value, as the GPU does."""
        f = _fp8(fmt)
        d = _dt(out_dtype)
        A = np.asarray(A)
        B = np.asarray(B)
        if A.dtype != np.uint8 or B.dtype != np.uint8:
            raise TypeError("oracle.gemm_fp8 takes uint8 FP8 patterns")
        if A.ndim != 2 or B.ndim != 2:
            raise ValueError("operands must be 2-D")
        if A.size and A.strides[1] != 1:
            A = np.ascontiguousarray(A)
        if B.size and B.strides[1] != 1:
            B = np.ascontiguousarray(B)
        M, K = A.shape
        N, Kb = B.shape
        if Kb != K:
            raise ValueError(f"K mismatch: {K} vs {Kb}")
        i0, i1 = rows if rows is not None else (0, M)
        j0, j1 = cols if cols is not None else (0, N)
        if not (0 <= i0 <= i1 <= M and 0 <= j0 <= j1 <= N):
            raise ValueError("rows/cols out of range")
        lda = A.strides[0] if A.shape[0] > 1 else max(A.shape[1], 1)
        ldb = B.strides[0] if B.shape[0] > 1 else max(B.shape[1], 1)
        out16 = np.zeros((i1 - i0, j1 - j0), dtype=np.uint16)
        out64 = np.zeros((i1 - i0, j1 - j0), dtype=np.float64) if want_f64 else None
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        a32 = float(np.float32(alpha))
        if out16.size:
            self._lib.oracle_gemm_fp8(A.ctypes.data_as(u8p) if A.size else None,
                                      B.ctypes.data_as(u8p) if B.size else None,
                                      M, N, K, lda, ldb, f, d, a32, i0, i1, j0, j1,
                                      out16.ctypes.data_as(u16p),
                                      out64.ctypes.data_as(f64p) if want_f64 else None, j1 - j0)
        return (out16, out64) if want_f64 else out16

    return fp8_to_double, gemm_fp8


Oracle.fp8_to_double, Oracle.gemm_fp8 = _fp8_methods()


def _row_stride(X: np.ndarray) -> int:
    return X.strides[0] if X.shape[0] > 1 else max(X.shape[1], 1)


def _mx_methods():
    def ue8m0_to_double(self, bits) -> np.ndarray:
        """Value 2^(x - 127) of each UE8M0 scale byte (NaN for 255)."""
        b = np.asarray(bits, dtype=np.uint8)
        return np.array([self._lib.oracle_ue8m0_to_double(int(v)) for v in b.ravel()],
                        dtype=np.float64).reshape(b.shape)

    def gemm_mx(self, A, B, SA, SB, *, fmt="e4m3", out_dtype="bf16", alpha=1.0, rows=None,
                cols=None, want_f64: bool = False):
        """Oracle block-scaled FP8 GEMM: D = round(alpha * sum_k (A[i,k] sa) (B[j,k] sb))
        with one UE8M0 scale per 32 K elements of each row: SA (M, ceil(K/32)) and
        SB (N, ceil(K/32)) uint8, row-major (row stride free, unit inner stride)."""
        f = _fp8(fmt)
        d = _dt(out_dtype)
        A, B, SA, SB = (np.asarray(x) for x in (A, B, SA, SB))
        for x in (A, B, SA, SB):
            if x.dtype != np.uint8 or x.ndim != 2:
                raise TypeError("oracle.gemm_mx takes 2-D uint8 patterns")
        A, B, SA, SB = (np.ascontiguousarray(x) if x.size and x.strides[1] != 1 else x
                        for x in (A, B, SA, SB))
        M, K = A.shape
        N, Kb = B.shape
        groups = -(-K // 32)
        if Kb != K:
            raise ValueError(f"K mismatch: {K} vs {Kb}")
        if SA.shape != (M, groups) or SB.shape != (N, groups):
            raise ValueError(f"scale shapes {SA.shape}, {SB.shape}; want ({M}, {groups}), "
                             f"({N}, {groups})")
        i0, i1 = rows if rows is not None else (0, M)
        j0, j1 = cols if cols is not None else (0, N)
        if not (0 <= i0 <= i1 <= M and 0 <= j0 <= j1 <= N):
            raise ValueError("rows/cols out of range")
        out16 = np.zeros((i1 - i0, j1 - j0), dtype=np.uint16)
        out64 = np.zeros((i1 - i0, j1 - j0), dtype=np.float64) if want_f64 else None
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        ptr = (lambda x: x.ctypes.data_as(u8p) if x.size else None)
        if out16.size:
            self._lib.oracle_gemm_mx(ptr(A), ptr(B), ptr(SA), ptr(SB), M, N, K,
                                     _row_stride(A), _row_stride(B), _row_stride(SA),
                                     _row_stride(SB), f, d, float(np.float32(alpha)),
                                     i0, i1, j0, j1, out16.ctypes.data_as(u16p),
                                     out64.ctypes.data_as(f64p) if want_f64 else None, j1 - j0)
        return (out16, out64) if want_f64 else out16

    return ue8m0_to_double, gemm_mx


Oracle.ue8m0_to_double, Oracle.gemm_mx = _mx_methods()

_lock = threading.Lock()
_default: Oracle | None = None


def get() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gemm(A, B, **kw):
    return get().gemm(A, B, **kw)


def to_double(bits, dtype):
    return get().to_double(bits, dtype)


def from_double(x, dtype):
    return get().from_double(x, dtype)


def num_threads() -> int:
    return get().num_threads()


def gemm_fp8(A, B, **kw):
    return get().gemm_fp8(A, B, **kw)


def fp8_to_double(bits, fmt):
    return get().fp8_to_double(bits, fmt)


def gemm_mx(A, B, SA, SB, **kw):
    return get().gemm_mx(A, B, SA, SB, **kw)


def ue8m0_to_double(bits):
    return get().ue8m0_to_double(bits)
