"""Buffers past 32-bit byte offsets and past the 1 GiB item limit.

The layouts cut every piece into items of at most 1 GiB (the Atoms count
16-byte vectors in 32 bits) and all offsets are 64-bit.  These tests drive
each kind of kernel over buffers of 2.25 to 4.5 GiB per rank, with ragged
sizes, in the default launch configuration:

* AllReduce bf16, 2 ranks x 2.5 GiB (+6 bytes), one-shot, two-shot, fused
  two-shot and ring; 3 ranks x 2.25 GiB (+6 bytes), ring (whose running sum
  then crosses stages as two 16-bit halves) and fused two-shot;
* ReduceScatter fp32, 2 ranks x 2.5 GiB (bulk path, 1.25 GiB outputs);
* AllGather u8, 2 ranks x 2.25 GiB (+5 bytes): outputs of 4.5 GiB, the second
  block at an odd offset;
* AllToAll u8, 2 ranks x 4.5 GiB (+2 bytes): odd-sized chunks, source
  offsets past 4 GiB.

Inputs are rotations of one seeded block (inputs.Tiled).  Outputs are
checked two ways: on the device, against properties that hold at any size
(all AllReduce outputs equal; every AllGather / AllToAll block equals its
source range, byte for byte); and element by element against the oracle at
a sample of positions -- a million random ones plus every position within
2048 elements of each GiB boundary, of 2^31 and 2^32 bytes, and of both
ends -- with the oracle run on the inputs at those positions (every
collective here is elementwise, so sampling commutes with it).
"""

import numpy as np
import pytest
import torch

import oracle
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from workload_inputs import Tiled
from gpu_util import Handle, RankBuffers, stream, sync

pytestmark = pytest.mark.gpu

GiB = 1 << 30
_TORCH = {"u8": torch.uint8, "bf16": torch.int16, "f32": torch.float32}
_NP = {"u8": np.uint8, "bf16": np.uint16, "f32": np.float32}
_E = {"u8": 1, "bf16": 2, "f32": 4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()
    yield
    torch.cuda.empty_cache()


def upload(buf, r, t, at=0):
    """Write Tiled `t` into rank buffer r starting at element `at`."""
    E = _E[t.dtype]
    v = buf.view(r)
    for start, chunk in t.chunks():
        b = np.ascontiguousarray(chunk).view(np.uint8)
        o = (at + start) * E
        v[o:o + b.size].copy_(torch.from_numpy(b))


def positions(n, E, seed, extra=()):
    """Sampled element positions in [0, n): random ones plus the boundaries."""
    rng = np.random.default_rng(seed)
    parts = [rng.integers(0, n, 1 << 20), np.arange(0, 4096), np.arange(n - 4096, n)]
    for edge in [k * GiB for k in range(1, 6)] + [1 << 31, 1 << 32] + list(extra):
        e = edge // E
        parts.append(np.arange(e - 2048, e + 2048))
    idx = np.unique(np.concatenate(parts).astype(np.int64))
    return idx[(idx >= 0) & (idx < n)]


def sample(buf, r, dtype, idx, at=0):
    """Elements of rank buffer r at positions at + idx (read on the device)."""
    t = buf.view(r)
    if dtype != "u8":
        t = t.view(_TORCH[dtype])
    got = t[torch.from_numpy(idx + at).to(t.device)].cpu().numpy()
    return got.view(_NP[dtype])


def as_bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.fixture(scope="module")
def ar_inputs():
    S = 5 * GiB // 2 + 6
    n = S // 2
    T = [Tiled(n, "bf16", seed=21 + r, shift=1001 * r) for r in range(2)]
    src = RankBuffers([S] * 2)
    for r in range(2):
        upload(src, r, T[r])
    yield S, n, T, src
    del src
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", [P.PL_LAYOUT_AUTO, P.PL_LAYOUT_TWO_SHOT, P.PL_LAYOUT_TWO_SHOT_FUSED,
                                    P.PL_LAYOUT_RING])
def test_all_reduce_2x2_5GiB(ar_inputs, layout):
    S, n, T, src = ar_inputs
    dst = RankBuffers([S] * 2)
    h = Handle(2)
    if layout:
        P.check(P.purlin_tune_override(h.h, {"layout": layout}))
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), S, P.PL_BF16, 0, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    assert torch.equal(dst.view(0), dst.view(1))
    pos = positions(n, 2, seed=31)
    want = oracle.all_reduce([t.at(pos) for t in T], "bf16")
    for r in range(2):
        assert np.array_equal(sample(dst, r, "bf16", pos), want[r]), r
    assert dst.guards_intact() and src.guards_intact()


@pytest.mark.parametrize("layout", [P.PL_LAYOUT_RING, P.PL_LAYOUT_TWO_SHOT_FUSED])
def test_all_reduce_3x2_25GiB(layout):
    """Three ranks: the ring's bf16 running sum travels as two 16-bit halves
    in the outputs, at offsets past 2^31 and 2^32 bytes."""
    world, S = 3, 9 * GiB // 4 + 6
    n = S // 2
    T = [Tiled(n, "bf16", seed=31 + r, shift=777 * r) for r in range(world)]
    src = RankBuffers([S] * world)
    for r in range(world):
        upload(src, r, T[r])
    dst = RankBuffers([S] * world)
    h = Handle(world)
    P.check(P.purlin_tune_override(h.h, {"layout": layout}))
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), S, P.PL_BF16, 0, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    assert torch.equal(dst.view(0), dst.view(1)) and torch.equal(dst.view(0), dst.view(2))
    pos = positions(n, 2, seed=37)
    want = oracle.all_reduce([t.at(pos) for t in T], "bf16")
    for r in range(world):
        assert np.array_equal(sample(dst, r, "bf16", pos), want[r]), r
    assert dst.guards_intact() and src.guards_intact()
    del src, dst
    torch.cuda.empty_cache()


def test_reduce_scatter_f32_2x2_5GiB():
    world, S = 2, 5 * GiB // 2
    n = S // 4
    c = n // world
    T = [Tiled(n, "f32", seed=41 + r, shift=333 * r) for r in range(world)]
    src = RankBuffers([S] * world)
    for r in range(world):
        upload(src, r, T[r])
    dst = RankBuffers([c * 4] * world)
    h = Handle(world)
    P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), S, P.PL_F32, 0, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    j = positions(c, 4, seed=43)
    # source s, laid out as `world` chunks of the sampled positions, in rank order
    a = [np.concatenate([T[s].at(r * c + j) for r in range(world)]) for s in range(world)]
    want = oracle.reduce_scatter(a, "f32")
    for r in range(world):
        assert np.array_equal(as_bits(sample(dst, r, "f32", j)), as_bits(want[r])), r
    assert dst.guards_intact()
    del src, dst
    torch.cuda.empty_cache()


def test_all_gather_u8_outputs_past_4GiB():
    world, S = 2, 9 * GiB // 4 + 5
    T = [Tiled(S, "u8", seed=51 + r, shift=77 * r) for r in range(world)]
    src = RankBuffers([S] * world)
    for r in range(world):
        upload(src, r, T[r])
    dst = RankBuffers([world * S] * world)
    h = Handle(world)
    P.check(P.purlin_all_gather(h.h, src.ptrs(), dst.ptrs(), S, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    for r in range(world):
        for s in range(world):
            assert torch.equal(dst.view(r)[s * S:(s + 1) * S], src.view(s)), (r, s)
    # output byte 2^32 falls in block 1
    j = positions(S, 1, seed=53, extra=[(1 << 32) - S])
    want = oracle.all_gather([t.at(j) for t in T])
    for r in range(world):
        got = np.concatenate([sample(dst, r, "u8", j, at=s * S) for s in range(world)])
        assert np.array_equal(got, want[r]), r
    assert dst.guards_intact()
    del src, dst
    torch.cuda.empty_cache()


def test_all_to_all_u8_sources_past_4GiB():
    world, S = 2, 9 * GiB // 2 + 2
    C = S // world
    T = [Tiled(S, "u8", seed=61 + r, shift=5 * r) for r in range(world)]
    src = RankBuffers([S] * world)
    for r in range(world):
        upload(src, r, T[r])
    dst = RankBuffers([S] * world)
    h = Handle(world)
    P.check(P.purlin_all_to_all(h.h, src.ptrs(), dst.ptrs(), S, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    for d in range(world):
        for s in range(world):
            assert torch.equal(dst.view(d)[s * C:(s + 1) * C], src.view(s)[d * C:(d + 1) * C]), (d, s)
    j = positions(C, 1, seed=63, extra=[(1 << 32) - C])
    a = [np.concatenate([T[s].at(d * C + j) for d in range(world)]) for s in range(world)]
    want = oracle.all_to_all(a)
    for d in range(world):
        got = np.concatenate([sample(dst, d, "u8", j, at=s * C) for s in range(world)])
        assert np.array_equal(got, want[d]), d
    assert dst.guards_intact()
    del src, dst
    torch.cuda.empty_cache()
