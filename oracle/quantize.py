"""Per-tensor FP8 (e4m3) quantisation with a power-of-two descale
(test infrastructure only).

ZYFA README, "Usage": ``fp8_quantize`` returns the e4m3 tensor and one
power-of-two descale per tensor; every conversion rounds to nearest even
("Kernel design").  The descale is the smallest power of two with
``max|x| / descale <= 448`` (448 = largest finite e4m3 value), 1 for an
all-zero tensor.  Each element becomes the e4m3 value nearest to
``x / descale`` (ties to the even code), saturated to +-448.

The encoder works from the value table of ``formats.e4m3_to_f64`` (the
format definition), not from any library conversion.  Pinned by
``tests/test_oracle.py::test_quantize_*``.
"""

from __future__ import annotations

import math

import numpy as np

from .formats import e4m3_to_f64

E4M3_MAX = 448.0

_POS_CODES = np.array([c for c in range(0x7F) if not np.isnan(e4m3_to_f64(np.uint8(c)))],
                      dtype=np.uint8)            # 0x00 .. 0x7E, ascending values
_POS_VALS = e4m3_to_f64(_POS_CODES)


def descale_of(amax: float) -> float:
    """Smallest power of two d with amax / d <= 448 (1.0 when amax == 0)."""
    if amax == 0.0:
        return 1.0
    k = math.ceil(math.log2(amax / E4M3_MAX))
    # guard the float64 log2 at exact boundaries
    while amax > E4M3_MAX * 2.0 ** k:
        k += 1
    while amax <= E4M3_MAX * 2.0 ** (k - 1):
        k -= 1
    return 2.0 ** k


def e4m3_encode_rne(y: np.ndarray) -> np.ndarray:
    """e4m3 codes of real values, round to nearest, ties to even, saturating."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), E4M3_MAX)
    hi = np.searchsorted(_POS_VALS, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS_VALS) - 1)
    lo = np.maximum(hi - 1, 0)
    vlo, vhi = _POS_VALS[lo], _POS_VALS[hi]
    dlo, dhi = a - vlo, vhi - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0))
    idx = np.where(a >= vhi, hi, np.where(pick_hi, hi, lo))
    codes = _POS_CODES[idx].astype(np.uint8)
    neg = (y < 0) | ((y == 0) & np.signbit(y))
    return np.where(neg, codes | np.uint8(0x80), codes).astype(np.uint8)


def fp8_quantize_f64(x: np.ndarray):
    """(codes, descale) of real values ``x`` (any shape)."""
    x = np.asarray(x, dtype=np.float64)
    amax = float(np.abs(x).max()) if x.size else 0.0
    d = descale_of(amax)
    return e4m3_encode_rne(x / d), d
