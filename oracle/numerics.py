"""Exact number-format conversions used by the oracle (test infrastructure only).

* bf16 -> float64 decode and float64 -> bf16 round-to-nearest-even (the GEMM's output
  conversion; the tilelang page only writes a cast of the fp32 accumulator to the output
  dtype in its epilogue, the round-to-nearest-even reading is the CUDA default cast).
* OCP E4M3FN decode (bias 7, no infinities, 0x7F/0xFF are NaN) and E8M0 decode
  (value 2**(byte - 127), 0xFF is NaN): the MXFP8 operand and scale formats of
  ``gemm_mxfp8_blockscaled_1d1d.py`` ("Blockscale size: (M, N, K) = (1, 1, 128)").

Everything is written from the format definitions with float64 arithmetic, which is
exact for every value these formats can hold.
"""
from __future__ import annotations

import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode raw bf16 bit patterns (uint16) to float64 exactly."""
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    sign = np.where(b & 0x8000, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    f = (b & 0x7F).astype(np.float64)
    normal = (1.0 + f / 128.0) * np.ldexp(1.0, (e - 127).astype(np.int64))
    sub = f * 2.0 ** -133
    val = np.where(e == 0, sub, normal)
    val = np.where(e == 255, np.where(f == 0, np.inf, np.nan), val)
    return sign * val


def f64_to_bf16_rne(x) -> np.ndarray:
    """Round float64 values to bf16 with round-half-to-even; returns uint16 bits.

    The rounding step (quantum) is 2**(e-7) for |x| in [2**e, 2**(e+1)) inside the normal
    range and 2**-133 below 2**-126; results above the largest bf16 become infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    m, e = np.frexp(a)  # a = m * 2**e with m in [0.5, 1)
    quantum_exp = np.where(a >= 2.0 ** -126, e.astype(np.int64) - 8, -133)
    q = np.ldexp(np.rint(np.ldexp(a, -quantum_exp)), quantum_exp)
    # encode q (a bf16 value or >= 2**128) to bits
    out = np.zeros(x.shape, dtype=np.int64)
    over = q > BF16_MAX
    sub = q < 2.0 ** -126
    out[sub] = np.rint(q[sub] * 2.0 ** 133).astype(np.int64)
    nrm = ~sub & ~over
    qm, qe = np.frexp(q[nrm])
    out[nrm] = ((qe.astype(np.int64) - 1 + 127) << 7) | np.rint((qm * 2.0 - 1.0) * 128.0).astype(np.int64)
    out[over] = 0x7F80
    out[np.isnan(x)] = 0x7FC0
    out = out | np.where(np.signbit(x), 0x8000, 0)
    return out.astype(np.uint16)


def e4m3fn_to_f64(codes) -> np.ndarray:
    """Decode OCP FP8 E4M3FN codes (uint8) to float64 exactly."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    f = (c & 0x7).astype(np.float64)
    normal = (1.0 + f / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int64))
    sub = f * 2.0 ** -9
    val = np.where(e == 0, sub, normal)
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def e8m0_to_f64(codes) -> np.ndarray:
    """Decode E8M0 scale bytes (uint8) to float64: 2**(byte - 127); 0xFF is NaN."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    val = np.ldexp(1.0, (c - 127).astype(np.int64))
    return np.where(c == 255, np.nan, val)
