"""Persistent elementwise add oracle (test infrastructure only).

helion "Implement persistent kernels", the ``_simple_add_kernel`` listings: every element of
the result is ``x + y`` in the inputs' dtype (fp32); the persistent tile loop only decides
which program writes which element, never the value.  numpy's float32 addition is the
IEEE-754 binary32 sum with round-to-nearest-even and gradual underflow, which is the value
every correct implementation must produce bit for bit.

The multi-loop listings of the same page scale each tile space by a constant
(``result1 = 2.0 * x``, ``result2 = 3.0 * y``): :func:`scale_f32` is that product, one
IEEE binary32 multiply per element.
"""
from __future__ import annotations

import numpy as np


def add_f32(x, y) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    y = np.asarray(y, dtype=np.float32)
    if x.shape != y.shape:
        raise ValueError("x and y must have the same shape")
    with np.errstate(over="ignore", invalid="ignore"):
        return np.add(x, y, dtype=np.float32)


def scale_f32(x, a: float) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        return np.multiply(x, np.float32(a), dtype=np.float32)
