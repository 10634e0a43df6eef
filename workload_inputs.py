"""Seeded synthetic inputs for the five collective workloads.

This module only draws numbers; it holds none of the collectives' arithmetic.
The CPU oracle, the GPU tests, the smoke check and the benchmark all take their
inputs from here, so both sides of every comparison see the same bytes.

Workloads (sizes are the defaults; every generator takes smaller sizes for
the parity tests):

  W1  AllReduce, 2 ranks, fp32, 1024 elements per rank, integers drawn
      uniformly from -8..8 inclusive and stored as fp32 (sums are exact), seed 0.
  W2  AllReduce, 8 ranks, bf16, 32 Mi elements (64 MiB) per rank, N(0,1), seed 1.
  W3  ReduceScatter, 8 ranks, 64 Mi elements per rank, U(-1,1), seed 2; fp32
      (256 MiB per rank) and bf16 (128 MiB per rank) from the same draw.
  W4  AllGather / AllToAll, 8 ranks, uint8 payload drawn uniformly from 0..255,
      per-rank size 1 KiB .. 256 MiB in powers of 4, seed 3 (a fresh generator
      per size).
  W5  AllToAllV / AllGatherV, 8 ranks, bf16 N(0,1) payload, element counts
      drawn uniformly from 0..4 Mi inclusive, seed 4, with a few counts forced
      afterwards so that the structure the workload names is always present:
      zero counts, counts that are not multiples of 8, a count of 1.

All draws use numpy's PCG64 (`default_rng`), rank-major.  bf16 data are the
fp32 draw rounded to nearest-even by torch's CPU conversion.
"""

from __future__ import annotations

import numpy as np
import torch

MI = 1 << 20


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of an fp32 draw, via torch's CPU rounding."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def w1_allreduce_ints(world: int = 2, n: int = 1024, seed: int = 0) -> np.ndarray:
    """(world, n) float32 holding integers from -8..8 inclusive."""
    rng = np.random.default_rng(seed)
    return rng.integers(-8, 9, size=(world, n)).astype(np.float32)


def w2_allreduce_bf16(world: int = 8, n: int = 32 * MI, seed: int = 1) -> np.ndarray:
    """(world, n) bf16 bit patterns (uint16) of N(0,1) draws."""
    rng = np.random.default_rng(seed)
    return to_bf16_bits(rng.standard_normal((world, n), dtype=np.float32))


def w3_reduce_scatter(world: int = 8, n: int = 64 * MI, seed: int = 2, dtype: str = "f32") -> np.ndarray:
    """(world, n) U(-1,1) draws, as float32 or as bf16 bit patterns."""
    rng = np.random.default_rng(seed)
    x = rng.random((world, n), dtype=np.float32)
    x *= np.float32(2.0)
    x -= np.float32(1.0)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return to_bf16_bits(x)
    raise ValueError(dtype)


W4_SIZES = [1 << (10 + 2 * k) for k in range(10)]  # 1 KiB .. 256 MiB, powers of 4


def w4_bytes(world: int = 8, size: int = 1 << 10, seed: int = 3) -> np.ndarray:
    """(world, size) uint8 payload."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(world, size), dtype=np.uint8)


def w5_counts(world: int = 8, max_count: int = 4 * MI, seed: int = 4):
    """Element counts for AllToAllV (world x world, [src][dst]) and AllGatherV (world).

    Forced entries (kept inside the drawn range):
      AllToAllV: C[0][1] = C[5][5] = 0, C[2][3] = max-1, C[7][0] = 13, C[3][6] = 1.
      AllGatherV: c[2] = 0, c[5] = max-3.
    Entries that do not exist for a smaller world are skipped.
    """
    rng = np.random.default_rng(seed)
    C = rng.integers(0, max_count + 1, size=(world, world)).astype(np.int64)
    c = rng.integers(0, max_count + 1, size=world).astype(np.int64)
    forced_c = [((0, 1), 0), ((5, 5), 0), ((2, 3), max(max_count - 1, 0)),
                ((7, 0), min(13, max_count)), ((3, 6), min(1, max_count))]
    for (s, d), v in forced_c:
        if s < world and d < world:
            C[s, d] = v
    for r, v in [(2, 0), (5, max(max_count - 3, 0))]:
        if r < world:
            c[r] = v
    return C, c


def w5_payloads(C: np.ndarray, c: np.ndarray, seed: int = 4):
    """bf16 payloads: per-rank AllToAllV send buffers, then AllGatherV buffers.

    Drawn after the counts from a generator seeded with [seed, 1].
    """
    rng = np.random.default_rng([seed, 1])
    world = len(c)
    a2av = [to_bf16_bits(rng.standard_normal(int(C[s].sum()), dtype=np.float32)) for s in range(world)]
    agv = [to_bf16_bits(rng.standard_normal(int(c[s]), dtype=np.float32)) for s in range(world)]
    return a2av, agv


class Tiled:
    """A rank buffer of `n` elements too large to draw element by element.

    One seeded block of `block` elements (N(0,1) for fp32 / bf16, 0..255 for
    uint8) is drawn once; element i of the buffer is
    block[(i + shift + 7 * (i // block)) % block], so every block-sized piece
    of the buffer is a different rotation of the draw.  `chunks()` yields the
    buffer piece by piece for upload; `at(idx)` gives the elements at chosen
    positions, so a test can evaluate the oracle on a sample of any buffer.
    """

    def __init__(self, n: int, dtype: str, seed: int, shift: int = 0, block: int = 16 * MI):
        self.n, self.dtype, self.shift, self.block = int(n), dtype, int(shift), int(block)
        rng = np.random.default_rng(seed)
        if dtype == "u8":
            self.base = rng.integers(0, 256, size=self.block, dtype=np.uint8)
        else:
            x = rng.standard_normal(self.block, dtype=np.float32)
            self.base = x if dtype == "f32" else to_bf16_bits(x)

    def at(self, idx: np.ndarray) -> np.ndarray:
        idx = np.asarray(idx, dtype=np.int64)
        return self.base[(idx + self.shift + 7 * (idx // self.block)) % self.block]

    def chunks(self):
        for j, start in enumerate(range(0, self.n, self.block)):
            m = min(self.block, self.n - start)
            o = (self.shift + 7 * j) % self.block
            yield start, np.concatenate((self.base[o:], self.base[:o]))[:m]
