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
    if len(tensors) != world:
        raise ValueError(f"{what}: expected {world} tensors (one per rank), got {len(tensors)}")
    for t in tensors:
        if not (t.is_cuda or t.is_pinned()) or not t.is_contiguous():
            raise ValueError(f"{what}: tensors must be contiguous CUDA tensors or pinned host tensors")


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
    _same(xs, handle.world, "all_reduce")
    _same(outs, handle.world, "all_reduce")
    dt = _DTYPES.get(xs[0].dtype)
    if dt is None or any(t.dtype != xs[0].dtype or t.numel() != xs[0].numel() for t in list(xs) + list(outs)):
        raise ValueError("all_reduce: float32 or bfloat16 tensors of one size")
    with _on(handle):
        _check(P.purlin_all_reduce(handle.raw, xs, outs, xs[0].numel() * xs[0].element_size(), dt, int(reduction_mode),
                                   _stream(stream, handle.device)), "all_reduce")


def reduce_scatter(xs, outs, handle: Handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    """outs[r] = chunk r (of world equal chunks along dim 0) of the sum of xs."""
    _same(xs, handle.world, "reduce_scatter")
    _same(outs, handle.world, "reduce_scatter")
    dt = _DTYPES.get(xs[0].dtype)
    if dt is None:
        raise ValueError("reduce_scatter: float32 or bfloat16 tensors")
    with _on(handle):
        _check(P.purlin_reduce_scatter(handle.raw, xs, outs, xs[0].numel() * xs[0].element_size(), dt,
                                       int(reduction_mode), _stream(stream, handle.device)), "reduce_scatter")


def all_gather(xs, outs, handle: Handle, stream=None):
    """outs[r] = concatenation of xs along dim 0, for every rank r."""
    _same(xs, handle.world, "all_gather")
    _same(outs, handle.world, "all_gather")
    with _on(handle):
        _check(P.purlin_all_gather(handle.raw, xs, outs, xs[0].numel() * xs[0].element_size(),
                                   _stream(stream, handle.device)), "all_gather")


def all_to_all(xs, outs, handle: Handle, stream=None):
    """outs[d] chunk s = xs[s] chunk d (world equal chunks along dim 0)."""
    _same(xs, handle.world, "all_to_all")
    _same(outs, handle.world, "all_to_all")
    with _on(handle):
        _check(P.purlin_all_to_all(handle.raw, xs, outs, xs[0].numel() * xs[0].element_size(),
                                   _stream(stream, handle.device)), "all_to_all")


def all_gather_v(xs, outs, handle: Handle, stream=None):
    """outs[r] = concatenation of all of xs (each rank's tensor in full), packed in rank order."""
    _same(xs, handle.world, "all_gather_v")
    with _on(handle):
        _check(P.purlin_all_gather_v(handle.raw, xs, outs, [t.numel() * t.element_size() for t in xs],
                                     _stream(stream, handle.device)), "all_gather_v")


def all_to_all_v(xs, outs, counts, handle: Handle, stream=None):
    """counts[s][d] elements go from rank s to rank d (packed, prefix-sum displacements)."""
    _same(xs, handle.world, "all_to_all_v")
    es = xs[0].element_size()
    flat = [int(c) * es for row in counts for c in row]
    with _on(handle):
        _check(P.purlin_all_to_all_v(handle.raw, xs, outs, flat, _stream(stream, handle.device)), "all_to_all_v")


def reduce_scatter_v(xs, outs, counts, handle: Handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    """outs[r] = the counts[r] elements of the sum starting at sum(counts[:r])."""
    _same(xs, handle.world, "reduce_scatter_v")
    dt = _DTYPES.get(xs[0].dtype)
    if dt is None:
        raise ValueError("reduce_scatter_v: float32 or bfloat16 tensors")
    es = xs[0].element_size()
    with _on(handle):
        _check(P.purlin_reduce_scatter_v(handle.raw, xs, outs, [int(c) * es for c in counts], dt, int(reduction_mode),
                                         _stream(stream, handle.device)), "reduce_scatter_v")
