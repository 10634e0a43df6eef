"""The checking build (libpurlin_gb_debug.so, compiled with PURLIN_DEBUG).

Every kernel tests each work item against the byte counts of the rank
buffers it touches before it moves any data.  First the checks must stay
silent on correct calls (results equal the oracle, status 0) on all three
kernels: register path, bulk ring, streamed copies.  Then
purlin_debug_limit_buffer makes one launch believe a buffer is shorter than
it is: the items past that point are skipped, the status reads
PL_ERR_BOUNDS, the bytes past the limit keep their old contents, and the next
call on the handle is correct again.  No access outside any buffer happens.
"""

import numpy as np
import pytest
import torch

import oracle
import workload_inputs as inputs
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle, RankBuffers, stream, sync

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(909)


@pytest.fixture
def checking():
    _build.build()
    P.load()
    lib = P.load_checking()
    with P.using(lib):
        yield lib


def bf16(n):
    return inputs.to_bf16_bits(RNG.standard_normal(n).astype(np.float32))


CASES = [
    ("register", {"path": P.PATH_REGISTER}),
    ("bulk", {"path": P.PATH_BULK}),
]


@pytest.mark.parametrize("name,tune", CASES)
def test_checks_are_silent_on_correct_calls(checking, name, tune):
    world = 8
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, tune))
        n = 8 * 30001
        ins = [bf16(n) for _ in range(world)]
        src = RankBuffers([n * 2] * world)
        src.upload(ins)
        dst = RankBuffers([n * 2] * world)
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        rs = RankBuffers([n // world * 2] * world)
        P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), rs.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        S = 65536 + 40
        xs = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        cs = RankBuffers([S] * world, [3, 0, 1, 0, 5, 0, 7, 0])
        cs.upload(xs)
        ag = RankBuffers([world * S] * world)
        P.check(P.purlin_all_gather(h.h, cs.ptrs(), ag.ptrs(), S, stream()))
        sync()
        assert h.status() == 0
        want = oracle.all_reduce(ins, "bf16")
        want_rs = oracle.reduce_scatter(ins, "bf16")
        flat = np.concatenate(xs)
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
            assert np.array_equal(rs.read(r, np.uint16), want_rs[r])
            assert np.array_equal(ag.read(r), flat)
        assert dst.guards_intact() and rs.guards_intact() and ag.guards_intact()
    finally:
        assert h.close() == P.PL_OK


@pytest.mark.parametrize("tune", [{"path": P.PATH_REGISTER},
                                  {"path": P.PATH_BULK},
                                  {"path": P.PATH_BULK, "schedule": P.PL_SCHED_QUEUE, "interleave_bytes": 8192},
                                  {"path": P.PATH_REGISTER, "layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 4096},
                                  {"path": P.PATH_REGISTER, "layout": P.PL_LAYOUT_RING, "chunk_bytes": 4096},
                                  {"path": P.PATH_REGISTER, "layout": P.PL_LAYOUT_TWO_SHOT_FUSED, "chunk_bytes": 4096}])
def test_limited_output_is_caught(checking, tune):
    world = 4
    n = 4 * 40000
    ins = [bf16(n) for _ in range(world)]
    src = RankBuffers([n * 2] * world)
    src.upload(ins)
    dst = RankBuffers([n * 2] * world)
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, tune))
        limit = n  # rank 2's output believed to hold half its bytes
        if tune.get("schedule") == P.PL_SCHED_QUEUE:
            # a copy: AllToAll with the same buffers
            dst.fill(0xEE)
            P.check(P.purlin_debug_limit_buffer(h.h, 1, 2, limit))
            P.check(P.purlin_all_to_all(h.h, src.ptrs(), dst.ptrs(), n * 2, stream()))
            sync()
            assert h.status() == P.PL_ERR_BOUNDS
            assert np.all(dst.read(2)[limit:] == 0xEE)   # chunks 2 and 3 of rank 2 lie past the limit
            assert dst.guards_intact()
            P.check(P.purlin_all_to_all(h.h, src.ptrs(), dst.ptrs(), n * 2, stream()))
            sync()
            assert h.status() == 0
            want = oracle.all_to_all([x.view(np.uint8) for x in ins])
            for r in range(world):
                assert np.array_equal(dst.read(r), want[r])
            return
        dst.fill(0xEE)
        P.check(P.purlin_debug_limit_buffer(h.h, 1, 2, limit))
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        sync()
        assert h.status() == P.PL_ERR_BOUNDS
        assert np.all(dst.read(2)[n * 2 - 64:] == 0xEE)      # the last bytes of rank 2 were never written
        assert dst.guards_intact()
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        sync()
        assert h.status() == 0
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK


def test_limited_input_is_caught(checking):
    world = 4
    n = 4 * 40000
    ins = [bf16(n) for _ in range(world)]
    src = RankBuffers([n * 2] * world)
    src.upload(ins)
    dst = RankBuffers([n // world * 2] * world)
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, {"path": P.PATH_BULK}))
        dst.fill(0xEE)
        P.check(P.purlin_debug_limit_buffer(h.h, 0, 1, 1000))
        P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        sync()
        assert h.status() == P.PL_ERR_BOUNDS
        assert dst.guards_intact()
        P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        sync()
        assert h.status() == 0
        want = oracle.reduce_scatter(ins, "bf16")
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK


def test_normal_build_accepts_the_hook():
    _build.build()
    P.load()
    h = Handle(2)
    try:
        assert P.purlin_debug_limit_buffer(h.h, 1, 0, 16) == P.PL_OK
        assert P.purlin_debug_limit_buffer(h.h, 1, 16, 16) == P.PL_ERR_INVALID_ARG
    finally:
        assert h.close() == P.PL_OK
