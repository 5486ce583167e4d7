"""fp64 GEMM oracle and the GEMM tolerance checks (test infrastructure only).

What the GEMM computes (tilelang "Introduce tile scheduler", the MXFP8 1x1x128
block-scaled kernel; tritonBLAS "Work Stealing Scheduler Kernel", the matmul entry
point): ``C = A . B`` with fp32 accumulation and a bf16 output.  The oracle computes the
exact-input product in fp64:

* bf16 operands decode exactly to fp64.
* MXFP8 operands: ``a[i, k] = e4m3(q[i, k]) * 2**(s[i, k // 128] - 127)``, exact in fp64
  (one E8M0 scale per row and 128-wide K block, "Blockscale size: (M, N, K) = (1, 1, 128)").
* ``C64 = A . B`` and ``Abs64 = |A| . |B|`` accumulate in fp64, k increasing (``gemm_f64.c``).
* ``Cref = bf16_rne(C64)``.

Checks (the bar these kernels are held to):

* (i)  relative Frobenius error ``||C - Cref||_F / ||Cref||_F <= 1e-3``.  Reading: the bar
  is taken against the bf16-rounded result, because bf16 output rounding alone already
  gives ~1.5e-3 relative Frobenius error against the unrounded fp64 product.
* (ii) per element ``|C - C64| <= 1e-2 * Abs64`` against the unrounded product.

Epilogue extension (tritonBLAS "Work Stealing Scheduler Kernel", the matmul hunk passes
``a_scale`` / ``b_scale`` "if quantized" and a bias marked TODO; their semantics are not on
the page).  Reading: per-tensor scales fold into one factor ``alpha = a_scale * b_scale`` and
the bias is one value per output column, so ``C = alpha * (A . B) + bias[n]``.  The bars
become: Frobenius against ``bf16_rne(alpha * C64 + bias)`` and, per element,
``|C - (alpha * C64 + bias)| <= 1e-2 * (|alpha| * Abs64 + |bias|)``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import numerics

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_f64.c")
_LIB = os.path.join(_HERE, "_gemm_f64.so")
_lib = None

FROB_TOL = 1e-3
ELEM_TOL = 1e-2


def build_library(force: bool = False) -> str:
    """Compile gemm_f64.c into a shared library next to it (plain gcc + OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_library())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_gemm_rows_f64.argtypes = [P, I64, P, I64, ctypes.c_int, I64, I64, P, I64, P, P]
        lib.oracle_gemm_entries_f64.argtypes = [P, I64, P, I64, ctypes.c_int, I64, P, P, I64, P, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


# ---------------------------------------------------------------------------- operands
def dequant_bf16(bits) -> np.ndarray:
    return numerics.bf16_bits_to_f64(bits)


def dequant_mxfp8(codes, scales) -> np.ndarray:
    """Rows x K e4m3 codes with rows x K/128 E8M0 scales -> exact fp64 values."""
    q = numerics.e4m3fn_to_f64(codes)
    s = numerics.e8m0_to_f64(scales)
    K = q.shape[1]
    return q * np.repeat(s, 128, axis=1)[:, :K]


# ------------------------------------------------------------------------------- GEMM
def _c64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def gemm_rows(A64, B64, b_kn: bool, K: int, N: int, rows) -> tuple[np.ndarray, np.ndarray]:
    """C64 and Abs64 for the listed rows of A (every column).  A: M x lda, B: see gemm_f64.c."""
    lib = _load()
    A64, B64 = _c64(A64), _c64(B64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    C = np.empty((rows.size, N), np.float64)
    Ca = np.empty((rows.size, N), np.float64)
    lib.oracle_gemm_rows_f64(A64.ctypes.data, A64.shape[1], B64.ctypes.data, B64.shape[1],
                             int(bool(b_kn)), N, K, rows.ctypes.data, rows.size,
                             C.ctypes.data, Ca.ctypes.data)
    return C, Ca


def gemm_full(A64, B64, b_kn: bool, M: int, N: int, K: int):
    return gemm_rows(A64, B64, b_kn, K, N, np.arange(M))


def gemm_entries(A64, B64, b_kn: bool, K: int, ii, jj) -> tuple[np.ndarray, np.ndarray]:
    lib = _load()
    A64, B64 = _c64(A64), _c64(B64)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    C = np.empty(ii.size, np.float64)
    Ca = np.empty(ii.size, np.float64)
    lib.oracle_gemm_entries_f64(A64.ctypes.data, A64.shape[1], B64.ctypes.data, B64.shape[1],
                                int(bool(b_kn)), K, ii.ctypes.data, jj.ctypes.data, ii.size,
                                C.ctypes.data, Ca.ctypes.data)
    return C, Ca


# ------------------------------------------------------------------------------ checks
def epilogue(C64, Abs64, alpha: float = 1.0, bias=None):
    """Apply ``C = alpha * C + bias[n]`` to the fp64 product and its error bound."""
    C = float(alpha) * np.asarray(C64, dtype=np.float64)
    A = abs(float(alpha)) * np.asarray(Abs64, dtype=np.float64)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)[None, :]
        C = C + b
        A = A + np.abs(b)
    return C, A


def check(C_bits, C64, Abs64, frob_tol: float = FROB_TOL, elem_tol: float = ELEM_TOL) -> dict:
    """Compare bf16 results (uint16 bits) with the fp64 oracle; raises AssertionError."""
    Cg = numerics.bf16_bits_to_f64(C_bits)
    Cref = numerics.bf16_bits_to_f64(numerics.f64_to_bf16_rne(C64))
    assert np.all(np.isfinite(Cg)), "non-finite GEMM output"
    num = float(np.linalg.norm((Cg - Cref).ravel()))
    den = float(np.linalg.norm(Cref.ravel()))
    frob = num / den if den > 0 else num
    err = np.abs(Cg - C64)
    bound = elem_tol * Abs64
    bad = err > bound
    worst = float(np.max(err / np.where(Abs64 > 0, Abs64, 1.0))) if err.size else 0.0
    info = {"frob_rel": frob, "worst_err_over_abs": worst, "n_bad": int(bad.sum()), "n": int(err.size)}
    assert frob <= frob_tol, f"relative Frobenius error {frob:.3e} > {frob_tol}: {info}"
    assert not bad.any(), f"{int(bad.sum())} elements exceed {elem_tol}*|A|.|B|: {info}"
    return info
