"""Torch-tensor front end over the C ABI, shaped like Purlin's Python API.

purlin 0.6.5 (PyPI page), Python section: `purlin.initialize(group, device,
arch, stream)` returns a handle, `purlin.all_reduce(x, out, handle, stream,
reduction_mode=...)` runs a collective, `purlin.finalize(handle, stream)`
frees the handle.  Here one process owns all ranks, so the "group" is just the
world size and every collective takes one tensor per rank.  Argument
marshalling only: checks shapes and dtypes, passes data pointers and byte
counts to libpurlin_gb.so and raises on a non-OK status.
"""

from __future__ import annotations

import enum

import torch

from . import purlin as P


class ReductionMode(enum.IntEnum):
    DETERMINISTIC = P.PL_DETERMINISTIC


_DTYPES = {torch.float32: P.PL_F32, torch.bfloat16: P.PL_BF16}


class Handle:
    def __init__(self, raw, world, device):
        self.raw, self.world, self.device = raw, world, device

    def __repr__(self):
        return f"purlin.Handle(world={self.world}, device={self.device})"


def _stream(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(status, what):
    if status != P.PL_OK:
        raise P.PurlinError(status, what)


def _on(handle):
    """Make the handle's device current for the call (the C ABI requires it)."""
    return torch.cuda.device(handle.device)


def _same(tensors, world, what):
    """One contiguous CUDA (or pinned host) tensor per rank."""
    if len(tensors) != world:
        raise ValueError(f"{what}: expected {world} tensors (one per rank), got {len(tensors)}")
    for t in tensors:
        if not t.is_contiguous():
            raise ValueError(f"{what}: tensors must be contiguous")


def _resident(tensors, what):
    for t in tensors:
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{what}: tensors must be CUDA tensors or pinned host tensors")


def _nbytes(t):
    return t.numel() * t.element_size()


def _sizes(tensors, want, what, side):
    """Each tensor holds exactly want[r] bytes (the library cannot see
    allocation sizes, so a short tensor would be written past its end)."""
    for r, (t, w) in enumerate(zip(tensors, want)):
        if _nbytes(t) != w:
            raise ValueError(f"{what}: {side}[{r}] holds {_nbytes(t)} bytes, the collective needs {w}")


def _one_dtype(tensors, dtype, what):
    if any(t.dtype != dtype for t in tensors):
        raise ValueError(f"{what}: every tensor must have dtype {dtype}")


def _checked(what, handle, xs, outs, in_bytes, out_bytes, reduce=False):
    """Argument checks shared by the collectives, all before any library call:
    one tensor per rank on each side, one dtype (float32 or bfloat16 for the
    reductions), the exact byte size of every input and output, residency."""
    _same(xs, handle.world, what)
    _same(outs, handle.world, what)
    dtype = xs[0].dtype
    _one_dtype(list(xs) + list(outs), dtype, what)
    dt = _DTYPES.get(dtype)
    if reduce and dt is None:
        raise ValueError(f"{what}: float32 or bfloat16 tensors")
    _sizes(xs, in_bytes, what, "inputs")
    _sizes(outs, out_bytes, what, "outputs")
    _resident(list(xs) + list(outs), what)
    return dt


def initialize(world: int, device=None, stream=None) -> Handle:
    """Create a handle for `world` ranks on `device` (default: current device)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        st, raw = P.purlin_initialize(world, None, 0, _stream(stream, device))
    _check(st, "initialize")
    return Handle(raw, world, device)


def finalize(handle: Handle, stream=None) -> None:
    st = P.purlin_finalize(handle.raw, _stream(stream, handle.device))
    handle.raw = None
    _check(st, "finalize")


def all_reduce(xs, outs, handle: Handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    """outs[r] = sum over s of xs[s], for every rank r (outs may be xs: in place)."""
    b = _nbytes(xs[0]) if len(xs) else 0
    dt = _checked("all_reduce", handle, xs, outs, [b] * handle.world, [b] * handle.world, reduce=True)
    with _on(handle):
        _check(P.purlin_all_reduce(handle.raw, xs, outs, b, dt, int(reduction_mode),
                                   _stream(stream, handle.device)), "all_reduce")


def reduce_scatter(xs, outs, handle: Handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    """outs[r] = chunk r (of world equal chunks along dim 0) of the sum of xs."""
    b = _nbytes(xs[0]) if len(xs) else 0
    if len(xs) and xs[0].numel() % handle.world:
        raise ValueError("reduce_scatter: the input length must split into world equal chunks")
    dt = _checked("reduce_scatter", handle, xs, outs, [b] * handle.world, [b // handle.world] * handle.world,
                  reduce=True)
    with _on(handle):
        _check(P.purlin_reduce_scatter(handle.raw, xs, outs, b, dt, int(reduction_mode),
                                       _stream(stream, handle.device)), "reduce_scatter")


def all_gather(xs, outs, handle: Handle, stream=None):
    """outs[r] = concatenation of xs along dim 0, for every rank r."""
    b = _nbytes(xs[0]) if len(xs) else 0
    _checked("all_gather", handle, xs, outs, [b] * handle.world, [handle.world * b] * handle.world)
    with _on(handle):
        _check(P.purlin_all_gather(handle.raw, xs, outs, b, _stream(stream, handle.device)), "all_gather")


def all_to_all(xs, outs, handle: Handle, stream=None):
    """outs[d] chunk s = xs[s] chunk d (world equal chunks along dim 0)."""
    b = _nbytes(xs[0]) if len(xs) else 0
    if len(xs) and xs[0].numel() % handle.world:
        raise ValueError("all_to_all: the length must split into world equal chunks")
    _checked("all_to_all", handle, xs, outs, [b] * handle.world, [b] * handle.world)
    with _on(handle):
        _check(P.purlin_all_to_all(handle.raw, xs, outs, b, _stream(stream, handle.device)), "all_to_all")


def all_gather_v(xs, outs, handle: Handle, stream=None):
    """outs[r] = concatenation of all of xs (each rank's tensor in full), packed in rank order."""
    _same(xs, handle.world, "all_gather_v")
    sizes = [_nbytes(t) for t in xs]
    _checked("all_gather_v", handle, xs, outs, sizes, [sum(sizes)] * handle.world)
    with _on(handle):
        _check(P.purlin_all_gather_v(handle.raw, xs, outs, sizes, _stream(stream, handle.device)), "all_gather_v")


def all_to_all_v(xs, outs, counts, handle: Handle, stream=None):
    """counts[s][d] elements go from rank s to rank d (packed, prefix-sum displacements)."""
    N = handle.world
    if len(counts) != N or any(len(row) != N for row in counts) or any(int(c) < 0 for row in counts for c in row):
        raise ValueError(f"all_to_all_v: counts must be {N} x {N} non-negative element counts")
    es = xs[0].element_size() if len(xs) else 1
    sent = [sum(int(c) for c in counts[s]) * es for s in range(N)]
    received = [sum(int(counts[s][d]) for s in range(N)) * es for d in range(N)]
    _checked("all_to_all_v", handle, xs, outs, sent, received)
    flat = [int(c) * es for row in counts for c in row]
    with _on(handle):
        _check(P.purlin_all_to_all_v(handle.raw, xs, outs, flat, _stream(stream, handle.device)), "all_to_all_v")


def reduce_scatter_v(xs, outs, counts, handle: Handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    """outs[r] = the counts[r] elements of the sum starting at sum(counts[:r])."""
    N = handle.world
    if len(counts) != N or any(int(c) < 0 for c in counts):
        raise ValueError(f"reduce_scatter_v: counts must be {N} non-negative element counts")
    es = xs[0].element_size() if len(xs) else 1
    total = sum(int(c) for c in counts) * es
    dt = _checked("reduce_scatter_v", handle, xs, outs, [total] * N, [int(c) * es for c in counts], reduce=True)
    with _on(handle):
        _check(P.purlin_reduce_scatter_v(handle.raw, xs, outs, [int(c) * es for c in counts], dt, int(reduction_mode),
                                         _stream(stream, handle.device)), "reduce_scatter_v")
