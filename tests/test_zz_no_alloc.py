"""The allocation-free AllReduce (purlin_all_reduce_noalloc) against the oracle.

purlin_all_reduce_noalloc serves callers that must not allocate device memory
once they run; its scratch is a fixed array inside the library, and its
kernel computes its own tiling and owner ranges instead of running a plan.
Called through the C ABI, two calls in a row (new inputs each time, the array
keeping the previous call's contents), every output element must equal the
oracle's ascending fold bit for bit -- the tolerance of every reduction test
here -- and the handle-based purlin_all_reduce's result too.  Also: the
full 8 x 64 MiB bf16 workload, ranks at different misalignments, in place,
the epoch wrap, a wait that runs out (through the test hook) and the size
limit.  This file is collected last so that a run stopping at the first
failure has run every other test first.
"""

import numpy as np
import pytest
import torch

import oracle
import workload_inputs as inputs
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle, RankBuffers, bits, stream, sync

pytestmark = pytest.mark.gpu

ESZ = {"f32": 4, "bf16": 2}
DT = {"f32": P.PL_F32, "bf16": P.PL_BF16}
NP = {"f32": np.float32, "bf16": np.uint16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


def _draw(rng, dtype, n):
    x = rng.standard_normal(n).astype(np.float32)
    return x if dtype == "f32" else inputs.to_bf16_bits(x)


def _status():
    return torch.full((1,), -1, dtype=torch.int32, device="cuda:0")


def _noalloc(world, src, dst, nbytes, dtype, status):
    P.check(P.purlin_all_reduce_noalloc(world, src.ptrs(), dst.ptrs(), nbytes, DT[dtype], status, stream()),
            "all_reduce_noalloc")


@pytest.mark.parametrize("dtype,world,n", [("bf16", 8, (1 << 20) + 7), ("f32", 5, 300001), ("bf16", 1, 4099),
                                           ("f32", 16, 4 * 65536 + 3), ("bf16", 3, 5)])
def test_noalloc_matches_oracle_two_calls_in_a_row(dtype, world, n):
    E = ESZ[dtype]
    rng = np.random.default_rng(99 + world)
    src = RankBuffers([n * E] * world)
    ref = RankBuffers([n * E] * world)
    out = RankBuffers([n * E] * world)
    status = _status()
    h = Handle(world)
    try:
        for call in range(2):
            ins = [_draw(rng, dtype, n) for _ in range(world)]
            src.upload(ins)
            out.fill(0)
            status.fill_(-1)
            _noalloc(world, src, out, n * E, dtype, status)
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), ref.ptrs(), n * E, DT[dtype], 0, stream()), "all_reduce")
            sync()
            assert int(status.item()) == P.PL_OK, call
            want = oracle.all_reduce(ins, dtype)
            for r in range(world):
                got = out.read(r, NP[dtype])
                assert np.array_equal(bits(got), bits(want[r])), (call, r)
                assert np.array_equal(bits(got), bits(ref.read(r, NP[dtype]))), (call, r)
            assert out.guards_intact() and src.guards_intact()
    finally:
        assert h.close() == P.PL_OK


def test_noalloc_full_workload_8x64MiB():
    """The headline shape: 8 ranks x 32 Mi bf16 N(0,1) elements (seed 1), every
    output element against the oracle, two calls in a row."""
    world, n = 8, 32 << 20
    x = inputs.w2_allreduce_bf16(world, n, seed=1)
    ins = [x[r] for r in range(world)]
    want = oracle.all_reduce(ins, "bf16")
    src = RankBuffers([n * 2] * world)
    out = RankBuffers([n * 2] * world)
    src.upload(ins)
    status = _status()
    for call in range(2):
        out.fill(0)
        status.fill_(-1)
        _noalloc(world, src, out, n * 2, "bf16", status)
        sync()
        assert int(status.item()) == P.PL_OK, call
        for r in range(world):
            assert np.array_equal(out.read(r, np.uint16), want[r]), (call, r)
    assert out.guards_intact() and src.guards_intact()
    del src, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_misaligned_ranks(dtype):
    """Every rank buffer at its own offset from a 16-byte boundary (multiples of
    the element size): sources not co-aligned take the element-wise fold,
    destinations at mixed residues take one copy per destination."""
    E = ESZ[dtype]
    world, n = 6, 200003
    rng = np.random.default_rng(5)
    for sm, dm in (([0, E, 2 * E, 3 * E, 4 * E, 5 * E], [E] * world),
                   ([4 * E] * world, [0, 2 * E, 4 * E, 6 * E, 8 * E, 10 * E])):
        sm = [m % 16 - (m % 16) % E for m in sm]
        dm = [m % 16 - (m % 16) % E for m in dm]
        src = RankBuffers([n * E] * world, sm)
        out = RankBuffers([n * E] * world, dm)
        ins = [_draw(rng, dtype, n) for _ in range(world)]
        src.upload(ins)
        status = _status()
        _noalloc(world, src, out, n * E, dtype, status)
        sync()
        assert int(status.item()) == P.PL_OK
        want = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert np.array_equal(bits(out.read(r, NP[dtype])), bits(want[r])), (sm, dm, r)
        assert out.guards_intact() and src.guards_intact()


def test_noalloc_in_place():
    """src[r] == dst[r]: each owner range is read in full before its sum is
    written, and the copies only write ranges already reduced."""
    world, n = 8, (1 << 20) + 11
    rng = np.random.default_rng(8)
    buf = RankBuffers([n * 2] * world)
    status = _status()
    for call in range(2):
        ins = [_draw(rng, "bf16", n) for _ in range(world)]
        buf.upload(ins)
        status.fill_(-1)
        _noalloc(world, buf, buf, n * 2, "bf16", status)
        sync()
        assert int(status.item()) == P.PL_OK
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(buf.read(r, np.uint16), want[r]), (call, r)
    assert buf.guards_intact()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Past 16384 tiles of 64 KiB the call returns PL_ERR_WORKSPACE before touching the GPU."""
    world = 8
    S = (16384 // world + 1) * (64 << 10) * world           # one tile per rank too many
    fake_src = [(1 << 44) + r * (1 << 34) for r in range(world)]
    fake_dst = [(1 << 45) + r * (1 << 34) for r in range(world)]
    assert P.purlin_all_reduce_noalloc(world, fake_src, fake_dst, S, P.PL_BF16, None, stream()) == P.PL_ERR_WORKSPACE
    assert P.purlin_all_reduce_noalloc(world, fake_src, fake_dst, 64 << 10, P.PL_U8, None, stream()) == \
        P.PL_ERR_UNSUPPORTED


def test_noalloc_across_the_epoch_wrap():
    """The scratch's epoch counter set near the end of its cycle: calls before,
    at and after the wrap all give the oracle's result.  The counter never
    holds 0xFFFFFFFF (the next launch would take epoch 0, the value of cleared
    flags), so the hook refuses it."""
    world, n, dtype = 8, (1 << 18) + 3, "bf16"
    rng = np.random.default_rng(7)
    assert P.purlin_debug_noalloc_set_epoch(0xFFFFFFFF, stream()) == P.PL_ERR_INVALID_ARG
    src = RankBuffers([n * 2] * world)
    out = RankBuffers([n * 2] * world)
    status = _status()
    P.check(P.purlin_debug_noalloc_set_epoch(0xFFFFFFFD, stream()))
    for call in range(4):
        ins = [_draw(rng, dtype, n) for _ in range(world)]
        src.upload(ins)
        out.fill(0)
        status.fill_(-1)
        _noalloc(world, src, out, n * 2, dtype, status)
        sync()
        assert int(status.item()) == P.PL_OK, call
        want = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert np.array_equal(out.read(r, np.uint16), want[r]), (call, r)


def test_noalloc_wait_runs_out_and_the_next_call_recovers():
    """The test hook drops the notify of owner 0's first tile and shortens the
    wait to 1 ms: its copy gives up, the status word reads PL_ERR_TIMEOUT and
    every CTA returns.  The next call (hook cleared) is complete and exact."""
    world, n = 4, (1 << 18) + 1
    rng = np.random.default_rng(11)
    src = RankBuffers([n * 2] * world)
    out = RankBuffers([n * 2] * world)
    status = _status()
    ins = [_draw(rng, "bf16", n) for _ in range(world)]
    src.upload(ins)
    assert P.purlin_debug_noalloc_next(1_000_000, 16384) == P.PL_ERR_INVALID_ARG
    P.check(P.purlin_debug_noalloc_next(1_000_000, 0))
    _noalloc(world, src, out, n * 2, "bf16", status)
    sync()
    assert int(status.item()) == P.PL_ERR_TIMEOUT
    status.fill_(-1)
    out.fill(0)
    _noalloc(world, src, out, n * 2, "bf16", status)
    sync()
    assert int(status.item()) == P.PL_OK
    want = oracle.all_reduce(ins, "bf16")
    for r in range(world):
        assert np.array_equal(out.read(r, np.uint16), want[r]), r
    assert out.guards_intact() and src.guards_intact()
