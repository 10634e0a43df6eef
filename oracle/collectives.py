"""Plain CPU statements of the collectives the datapath runs (test infrastructure).

Sources, by page and section:
  [NKI]  AWS Neuron NKI, "Collective Communication Kernels API Reference":
         the worked all-reduce example; "Background" (all-reduce sums tensors
         across ranks, all-gather gathers along dim 0, reduce-scatter sums then
         scatters dim-0 chunks, all-to-all exchanges dim-0 chunks); the
         all_to_all_hbm_kernel entry (rank i receives chunk i of every input).
  [PUR]  Purlin README (purlin 0.6.4 PKG-INFO), summary paragraph: the
         collectives are AllReduce, AllGather, ReduceScatter, AllToAll and
         variable-length variants of the last three; the datapath primitives are
         copy and N-to-1 reduce.  "Reduction determinism": deterministic mode
         gives bit-repeatable results for the same inputs.

Readings taken where the pages leave a step open:
  * Reductions accumulate in IEEE binary32, as a left fold in ascending rank
    order that starts from rank 0's value (not from +0.0), one rounding per add;
    bf16 results are rounded once, at the end, to nearest with ties to even.
  * ReduceScatter / AllToAll split dim 0 into `world` equal chunks; a size that
    does not split evenly is an error.
  * AllToAll places the chunk received from rank s at output chunk s.
  * The V variants take per-rank (AllGatherV, ReduceScatterV) or per
    (source, destination) pair (AllToAllV) element counts; data are packed
    with prefix-sum displacements in rank order.

Conventions: a "rank buffer" is a 1-D numpy array.  Floating-point data are
passed as float32 arrays ("f32") or as uint16 arrays holding bf16 bit patterns
("bf16").  Copy collectives do not look at values; they move elements of any
dtype exactly.  Every function returns a new list with one array per rank.

Pure numpy; nothing here is shared with, or calls, the CUDA library.
"""

from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# bf16 <-> fp32.  bf16 is the upper half of an IEEE binary32 pattern, so
# widening is exact and narrowing is a rounding of the dropped 16 bits.
# --------------------------------------------------------------------------


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening: the bf16 pattern becomes the top 16 bits of a binary32."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 bit patterns, nearest with ties to even.

    Written from the IEEE-754 rule: keep the top 16 bits; if the dropped
    16 bits are more than half an ulp, or exactly half and the kept pattern is
    odd, step the kept pattern up by one.  Because finite binary32 patterns of
    one sign are ordered like their integers, stepping up carries correctly
    into the exponent and turns the largest finite magnitude into infinity.
    NaNs stay NaN (quiet bit set); their payload bits are not pinned.
    """
    u = np.asarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    kept = (u >> np.uint32(16)).astype(np.uint32)
    dropped = u & np.uint32(0xFFFF)
    half = np.uint32(0x8000)
    round_up = (dropped > half) | ((dropped == half) & ((kept & np.uint32(1)) == 1))
    out = kept + round_up.astype(np.uint32)
    is_nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    out = np.where(is_nan, kept | np.uint32(0x0040), out)
    return out.astype(np.uint16).reshape(np.shape(x))


def _widen(buf: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        if buf.dtype != np.float32:
            raise TypeError("f32 rank buffers must be float32 arrays")
        return buf
    if dtype == "bf16":
        if buf.dtype != np.uint16:
            raise TypeError("bf16 rank buffers must be uint16 bit-pattern arrays")
        return bf16_bits_to_f32(buf)
    raise ValueError(f"reductions take f32 or bf16, not {dtype!r}")


def _narrow(acc: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return acc.astype(np.float32, copy=True)
    return f32_to_bf16_rne(acc)


def fold_sum(columns: list[np.ndarray]) -> np.ndarray:
    """Left fold in ascending rank order, binary32, one rounding per add.

    acc = columns[0]; then acc = fl32(acc + columns[s]) for s = 1 .. N-1.
    numpy adds two float32 arrays in float32 with round-to-nearest-even and
    without flushing subnormals, which is exactly the IEEE operation.
    """
    if not columns:
        raise ValueError("a reduction needs at least one rank")
    acc = np.array(columns[0], dtype=np.float32, copy=True)
    for col in columns[1:]:
        acc = np.add(acc, col, dtype=np.float32)
    return acc


def _check_ranks(inputs: list[np.ndarray]) -> int:
    world = len(inputs)
    if world < 1:
        raise ValueError("world must be at least 1")
    return world


# --------------------------------------------------------------------------
# Reductions (N-to-1 reduce).  [NKI] all_reduce_hbm_kernel, reduce_scatter_hbm_kernel.
# --------------------------------------------------------------------------


def all_reduce(inputs: list[np.ndarray], dtype: str) -> list[np.ndarray]:
    """Every rank receives the element-wise sum of all ranks' buffers."""
    world = _check_ranks(inputs)
    n = inputs[0].size
    if any(b.size != n for b in inputs):
        raise ValueError("all-reduce buffers must have equal length")
    total = _narrow(fold_sum([_widen(b, dtype) for b in inputs]), dtype)
    return [total.copy() for _ in range(world)]


def reduce_scatter(inputs: list[np.ndarray], dtype: str) -> list[np.ndarray]:
    """Sum, then rank r keeps dim-0 chunk r of the sum (world equal chunks)."""
    world = _check_ranks(inputs)
    n = inputs[0].size
    if any(b.size != n for b in inputs):
        raise ValueError("reduce-scatter buffers must have equal length")
    if n % world:
        raise ValueError("reduce-scatter length must split into world equal chunks")
    chunk = n // world
    out = []
    for r in range(world):
        cols = [_widen(b[r * chunk:(r + 1) * chunk], dtype) for b in inputs]
        out.append(_narrow(fold_sum(cols), dtype))
    return out


def reduce_scatter_v(inputs: list[np.ndarray], counts: list[int], dtype: str) -> list[np.ndarray]:
    """ReduceScatter with uneven chunks: rank r keeps counts[r] elements.

    Chunk r starts at the sum of counts[0..r-1] in every rank's buffer.
    """
    world = _check_ranks(inputs)
    if len(counts) != world or any(int(c) < 0 for c in counts):
        raise ValueError("need one non-negative count per rank")
    n = inputs[0].size
    if any(b.size != n for b in inputs) or sum(int(c) for c in counts) != n:
        raise ValueError("counts must cover each rank buffer exactly")
    out, start = [], 0
    for r in range(world):
        c = int(counts[r])
        cols = [_widen(b[start:start + c], dtype) for b in inputs]
        out.append(_narrow(fold_sum(cols), dtype))
        start += c
    return out


# --------------------------------------------------------------------------
# Copies.  [NKI] all_gather_hbm_kernel, all_to_all_hbm_kernel; [PUR] V variants.
# --------------------------------------------------------------------------


def all_gather(inputs: list[np.ndarray]) -> list[np.ndarray]:
    """Every rank receives all ranks' buffers stacked along dim 0, rank order."""
    world = _check_ranks(inputs)
    n = inputs[0].size
    if any(b.size != n for b in inputs):
        raise ValueError("all-gather buffers must have equal length")
    gathered = np.concatenate([np.asarray(b).reshape(-1) for b in inputs])
    return [gathered.copy() for _ in range(world)]


def all_to_all(inputs: list[np.ndarray]) -> list[np.ndarray]:
    """Rank d receives chunk d of every rank s, placed at chunk s of its output."""
    world = _check_ranks(inputs)
    n = inputs[0].size
    if any(b.size != n for b in inputs):
        raise ValueError("all-to-all buffers must have equal length")
    if n % world:
        raise ValueError("all-to-all length must split into world equal chunks")
    c = n // world
    out = []
    for d in range(world):
        dst = np.empty(n, dtype=inputs[0].dtype)
        for s in range(world):
            dst[s * c:(s + 1) * c] = inputs[s][d * c:(d + 1) * c]
        out.append(dst)
    return out


def all_gather_v(inputs: list[np.ndarray], counts: list[int]) -> list[np.ndarray]:
    """Every rank receives the first counts[s] elements of each rank s, packed."""
    world = _check_ranks(inputs)
    if len(counts) != world or any(int(c) < 0 for c in counts):
        raise ValueError("need one non-negative count per rank")
    for b, c in zip(inputs, counts):
        if int(c) > b.size:
            raise ValueError("count exceeds the rank buffer")
    gathered = np.concatenate([np.asarray(b).reshape(-1)[:int(c)] for b, c in zip(inputs, counts)])
    return [gathered.copy() for _ in range(world)]


def all_to_all_v(inputs: list[np.ndarray], counts) -> list[np.ndarray]:
    """counts[s][d] elements go from rank s to rank d.

    Rank s sends its block for d from offset sum(counts[s][:d]); rank d stores
    the block from s at offset sum(counts[:s][d]).
    """
    world = _check_ranks(inputs)
    C = [[int(v) for v in row] for row in counts]
    if len(C) != world or any(len(row) != world for row in C):
        raise ValueError("counts must be world x world")
    if any(v < 0 for row in C for v in row):
        raise ValueError("counts must be non-negative")
    for s in range(world):
        if sum(C[s]) > inputs[s].size:
            raise ValueError("send counts exceed the rank buffer")
    out = []
    for d in range(world):
        total = sum(C[s][d] for s in range(world))
        dst = np.empty(total, dtype=inputs[0].dtype)
        recv = 0
        for s in range(world):
            send = sum(C[s][:d])
            dst[recv:recv + C[s][d]] = inputs[s][send:send + C[s][d]]
            recv += C[s][d]
        out.append(dst)
    return out
