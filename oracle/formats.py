"""Exact float64 values of the stored input formats (test infrastructure only).

The oracle reads every input as the exact real number its bits encode, so an
FP8 input enters the float64 attention as ``code value x descale`` with no
rounding (ZYFA README, "Accuracy": error is measured "against fp64 attention on
the same quantized inputs").

* BF16: the upper 16 bits of an IEEE-754 binary32.
* e4m3 (``float8_e4m3fn``; ZYFA README, "Supported configurations": "4 exponent
  and 3 mantissa bits"): sign bit 7, biased exponent bits 6..3 (bias 7),
  mantissa bits 2..0.  Exponent field 0 encodes subnormals ``m/8 * 2**-6``;
  fields 1..15 encode ``(1 + m/8) * 2**(e-7)``; the two codes with every
  exponent and mantissa bit set (0x7F, 0xFF) are NaN, and there is no
  infinity.  Largest finite value 448, smallest normal 2**-6 (the README's
  "Clock speed and input values" section), smallest subnormal 2**-9.

Pinned by ``tests/test_oracle.py::test_e4m3_*`` and ``test_bf16_*``.
"""

from __future__ import annotations

import numpy as np


def bf16_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact float64 value of BF16 bit patterns given as uint16 (or int16)."""
    c = np.asarray(codes).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return c.view(np.float32).astype(np.float64)


def _e4m3_table() -> np.ndarray:
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if (code >> 7) & 1 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3 = _e4m3_table()


def e4m3_to_f64(codes: np.ndarray, descale: float = 1.0) -> np.ndarray:
    """Exact float64 value of e4m3 codes (uint8) times a per-tensor descale.

    The descale is a power of two (ZYFA README, "Usage": ``fp8_quantize``
    returns "one power-of-two scale per tensor"), so the product is exact.
    """
    return _E4M3[np.asarray(codes).astype(np.uint8)] * float(descale)
