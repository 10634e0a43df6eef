"""Distance in units in the last place between two arrays of one floating type.

Each value's bit pattern is mapped to an integer that grows with the value:
the pattern itself for +0 and positive values, minus its magnitude bits for
negative ones, so +0 and -0 both map to 0 and neighbouring representable
values map to neighbouring integers.  The distance of two values is the
difference of their integers.  Used to report how far a result lies from the
ascending-rank fold (0 everywhere means bit-identical, signed zeros apart).
"""

from __future__ import annotations

import numpy as np


def ordered(a: np.ndarray) -> np.ndarray:
    """Sign-folded ordered integers of float32 arrays or of uint16 bf16 patterns."""
    a = np.asarray(a)
    if a.dtype == np.float32:
        u = a.view(np.uint32).astype(np.int64)
        sign, mag = u >> 31, u & 0x7FFFFFFF
    elif a.dtype == np.uint16:
        u = a.astype(np.int64)
        sign, mag = u >> 15, u & 0x7FFF
    else:
        raise TypeError("float32 values or uint16 bf16 patterns")
    return np.where(sign == 1, -mag, mag)


def max_ulp(got: np.ndarray, want: np.ndarray) -> int:
    """Largest ulp distance between corresponding elements (0 for empty arrays)."""
    if np.asarray(got).size == 0:
        return 0
    return int(np.max(np.abs(ordered(got) - ordered(want))))
