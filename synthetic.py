"""Seeded synthetic inputs for the persistent GEMM and the persistent add.

This module is the only code shared by the CUDA path's callers (tests, bench,
smoke) and the CPU oracle's callers.  It draws random numbers and rounds them to
the storage type the kernels read; it holds none of the method's arithmetic
(no GEMM, no add, no scheduling, no output rounding).

Recipe (all draws use ``numpy.random.default_rng(seed)`` in float64, row-major):

* bf16 GEMM: draw A (M x K), then B as the K x N matrix of ``C = A . B``; round
  each to bf16 with round-to-nearest-even directly from float64.  When B is
  stored N x K ("K-major") the same K x N draw is transposed, so both layouts
  hold identical values.
* MXFP8 GEMM: draw A's payload (M x K, N(0,1)), A's scale exponents
  (M x K/128, uniform integers in [-4, 4]), then B's payload (N x K) and B's
  scale exponents (N x K/128).  Payloads are rounded to E4M3FN with
  round-to-nearest-even and saturation to +-448; scale bytes are E8M0
  (byte = 127 + exponent).
* add: draw x, then y, both N(0,1), rounded to float32 (numpy's RNE cast).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "f64_to_bf16_bits",
    "f64_to_e4m3_codes",
    "gemm_bf16_inputs",
    "gemm_mxfp8_inputs",
    "add_inputs",
]


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bfloat16 (RNE) and return the raw uint16 bits.

    Works on the float64 bit pattern: the 52-bit fraction is cut to 7 bits with
    round-half-to-even, then the exponent is re-biased from 1023 to 127.
    Magnitudes below 2**-126 take the bf16 subnormal grid (step 2**-133).
    Inputs must be finite.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("bf16 input rounding expects finite values")
    bits = x.view(np.uint64)
    sign = ((bits >> np.uint64(63)).astype(np.uint16)) << np.uint16(15)
    mag = bits & np.uint64(0x7FFF_FFFF_FFFF_FFFF)
    # round the fraction at bit 45: add 0x0FFF.. + lsb, then shift
    lsb = (mag >> np.uint64(45)) & np.uint64(1)
    r = (mag + np.uint64((1 << 44) - 1) + lsb) >> np.uint64(45)
    exp = (r >> np.uint64(7)).astype(np.int64) - 1023 + 127
    frac = (r & np.uint64(0x7F)).astype(np.int64)
    out = np.where(exp >= 255, 0x7F80, (np.clip(exp, 0, 254) << 7) | frac).astype(np.int64)
    # subnormal range of bf16 (and zero): |x| < 2**-126 -> multiples of 2**-133
    tiny = mag.view(np.float64) < 2.0 ** -126
    if np.any(tiny):
        q = np.rint(mag.view(np.float64)[tiny] * 2.0 ** 133).astype(np.int64)
        out[tiny] = q
    return (out.astype(np.uint16) | sign).astype(np.uint16)


def f64_to_e4m3_codes(x) -> np.ndarray:
    """Round float64 values to OCP E4M3FN codes (RNE, saturate to +-448)."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("e4m3 input rounding expects finite values")
    a = np.abs(x)
    m, e = np.frexp(a)  # a = m * 2**e, m in [0.5, 1)
    unb = e.astype(np.int64) - 1  # a = (2m) * 2**unb, 2m in [1, 2)
    step_exp = np.where(a >= 2.0 ** -6, unb - 3, -9)  # 3 fraction bits; subnormal step 2**-9
    q = np.rint(np.ldexp(a, -step_exp)) * np.ldexp(1.0, step_exp)
    q = np.minimum(q, 448.0)
    codes = np.zeros(x.shape, dtype=np.int64)
    sub = q < 2.0 ** -6
    codes[sub] = np.rint(q[sub] * 2.0 ** 9).astype(np.int64)
    nm = ~sub
    qm, qe = np.frexp(q[nm])
    E = qe.astype(np.int64) - 1
    frac = np.rint((qm * 2.0 - 1.0) * 8.0).astype(np.int64)
    codes[nm] = ((E + 7) << 3) | frac
    codes = codes | np.where(np.signbit(x), 0x80, 0)
    return codes.astype(np.uint8)


def _draw(rng, dist: str, shape, scale: float = 1.0) -> np.ndarray:
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape)
    if dist == "normal":
        return rng.standard_normal(size=shape) * scale
    raise ValueError(f"unknown distribution {dist!r}")


def gemm_bf16_inputs(M: int, N: int, K: int, seed: int, dist: str = "uniform",
                     b_layout: str = "kn", scale: float | None = None,
                     lda: int | None = None, ldb: int | None = None):
    """bf16 GEMM operands as uint16 bit arrays.

    Returns ``(A_bits, B_bits)``: A is M x lda (the first K columns hold data,
    padding columns are zero), B is K x ldb for ``b_layout == "kn"`` or N x ldb
    for ``"nk"``.  ``dist`` is "uniform" (U[-1,1]) or "normal"
    (N(0,1) * scale, default scale 1/sqrt(K)).
    """
    rng = np.random.default_rng(seed)
    if scale is None:
        scale = 1.0 / np.sqrt(K) if dist == "normal" else 1.0
    a = f64_to_bf16_bits(_draw(rng, dist, (M, K), scale))
    b = f64_to_bf16_bits(_draw(rng, dist, (K, N), scale))
    if b_layout == "nk":
        b = np.ascontiguousarray(b.T)
    elif b_layout != "kn":
        raise ValueError("b_layout must be 'kn' or 'nk'")
    lda = K if lda is None else lda
    A = np.zeros((M, lda), np.uint16)
    A[:, :K] = a
    inner_b = b.shape[1]
    ldb = inner_b if ldb is None else ldb
    B = np.zeros((b.shape[0], ldb), np.uint16)
    B[:, :inner_b] = b
    return A, B


def gemm_mxfp8_inputs(M: int, N: int, K: int, seed: int, exp_range: int = 4):
    """MXFP8 operands: (A_codes M x K u8, SFA M x K/128 u8, B_codes N x K u8, SFB N x K/128 u8)."""
    if K % 128:
        raise ValueError("MXFP8 operands need K % 128 == 0")
    rng = np.random.default_rng(seed)
    kb = K // 128
    a = f64_to_e4m3_codes(rng.standard_normal(size=(M, K)))
    sa = (127 + rng.integers(-exp_range, exp_range + 1, size=(M, kb))).astype(np.uint8)
    b = f64_to_e4m3_codes(rng.standard_normal(size=(N, K)))
    sb = (127 + rng.integers(-exp_range, exp_range + 1, size=(N, kb))).astype(np.uint8)
    return a, sa, b, sb


def add_inputs(rows: int, cols: int, seed: int):
    """fp32 x, y of shape rows x cols, each N(0,1), x drawn first."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=(rows, cols)).astype(np.float32)
    y = rng.standard_normal(size=(rows, cols)).astype(np.float32)
    return x, y


def gemm_bf16_sequence(shapes, seed: int, dist: str = "uniform"):
    """Several bf16 GEMM operand pairs drawn from ONE seeded stream, in the order given:
    A_0, B_0 (K x N), A_1, B_1, ...  Returns a list of (A_bits, B_bits)."""
    rng = np.random.default_rng(seed)
    out = []
    for (M, N, K) in shapes:
        scale = 1.0 / np.sqrt(K) if dist == "normal" else 1.0
        a = f64_to_bf16_bits(_draw(rng, dist, (M, K), scale))
        b = f64_to_bf16_bits(_draw(rng, dist, (K, N), scale))
        out.append((a, b))
    return out
