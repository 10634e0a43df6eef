"""Second, independent statement of the collectives: pure-Python per-element loops.

Used only to pin the numpy oracle on tiny inputs.  It shares nothing with the
oracle: binary32 rounding comes from Python's `struct` ('f' format, which
rounds a double to the nearest float, ties to even), and bf16 rounding picks
the nearer of the two neighbouring bf16 values by comparing distances.

Adding two binary32 values in binary64 and rounding the result to binary32
gives the correctly rounded binary32 sum, because binary64 carries more than
twice binary32's precision plus two bits (the classical double-rounding
condition), so `f32(a + b)` below is the IEEE binary32 add.
"""

from __future__ import annotations

import math
import struct


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def bits_f32(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def bf16_value(h: int) -> float:
    return bits_f32((h & 0xFFFF) << 16)


def bf16_round(x: float) -> int:
    """Nearest bf16 pattern to the binary32 value x, ties to the even pattern."""
    u = f32_bits(x)
    if math.isnan(x):
        return ((u >> 16) | 0x40) & 0xFFFF
    low = u >> 16                      # truncation toward zero
    if (u & 0xFFFF) == 0:
        return low
    high = low + 1                     # next pattern away from zero
    a, b = bf16_value(low), bf16_value(high)
    da, db = abs(x - a), abs(b - x)    # exact: all three share a binade or are adjacent
    if math.isinf(b):
        # the step above the largest finite bf16: infinity wins from the midpoint up
        mid_bits = (low << 16) | 0x8000
        mid = bits_f32(mid_bits)
        if abs(x) > abs(mid) or (abs(x) == abs(mid) and (low & 1)):
            return high
        return low
    if da < db:
        return low
    if db < da:
        return high
    return low if (low & 1) == 0 else high


def reduce_elem(vals: list[float], dtype: str):
    """Ascending-rank fold of one element position; returns a float (f32) or a bf16 pattern."""
    acc = f32(vals[0])
    for v in vals[1:]:
        acc = f32(acc + v)
    if dtype == "f32":
        return acc
    return bf16_round(acc)


def _widen(v, dtype):
    return float(v) if dtype == "f32" else bf16_value(int(v))


def all_reduce(ins, dtype):
    N, n = len(ins), len(ins[0])
    res = [reduce_elem([_widen(ins[s][i], dtype) for s in range(N)], dtype) for i in range(n)]
    return [list(res) for _ in range(N)]


def reduce_scatter(ins, dtype):
    N, n = len(ins), len(ins[0])
    c = n // N
    return [[reduce_elem([_widen(ins[s][r * c + j], dtype) for s in range(N)], dtype) for j in range(c)]
            for r in range(N)]


def reduce_scatter_v(ins, counts, dtype):
    N = len(ins)
    out = []
    for r in range(N):
        base = sum(counts[:r])
        out.append([reduce_elem([_widen(ins[s][base + j], dtype) for s in range(N)], dtype)
                    for j in range(counts[r])])
    return out


def all_gather(ins):
    N = len(ins)
    flat = [x for s in range(N) for x in ins[s]]
    return [list(flat) for _ in range(N)]


def all_to_all(ins):
    N, n = len(ins), len(ins[0])
    c = n // N
    out = [[None] * n for _ in range(N)]
    for s in range(N):
        for d in range(N):
            for j in range(c):
                out[d][s * c + j] = ins[s][d * c + j]
    return out


def all_gather_v(ins, counts):
    N = len(ins)
    flat = [ins[s][j] for s in range(N) for j in range(counts[s])]
    return [list(flat) for _ in range(N)]


def all_to_all_v(ins, C):
    N = len(ins)
    out = [[] for _ in range(N)]
    for d in range(N):
        for s in range(N):
            off = sum(C[s][k] for k in range(d))
            out[d].extend(ins[s][off:off + C[s][d]])
    return out
