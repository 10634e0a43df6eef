"""The allocation-free AllReduce (purlin_all_reduce_noalloc) against the handle-based one.

purlin_all_reduce_noalloc serves callers that must not allocate device memory
once they run; its scratch is a fixed array inside the library.  Called
through the C ABI, two calls in a row (new inputs each time, the array
keeping the previous call's contents), its outputs must equal
purlin_all_reduce's bit for bit, which is the tolerance of every reduction test
here.  This file is collected last so that a run stopping at the first failure
has run every other test first.
"""

import numpy as np
import pytest
import torch

from collective_datapath_reduce_gb300 import _build, inputs
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


@pytest.mark.parametrize("dtype,world,n", [("bf16", 8, (1 << 20) + 7), ("f32", 5, 300001), ("bf16", 1, 4099)])
def test_noalloc_matches_all_reduce_two_calls_in_a_row(dtype, world, n):
    E = ESZ[dtype]
    rng = np.random.default_rng(99 + world)
    src = RankBuffers([n * E] * world)
    ref = RankBuffers([n * E] * world)
    out = RankBuffers([n * E] * world)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda:0")
    h = Handle(world)
    try:
        for call in range(2):
            src.upload([_draw(rng, dtype, n) for _ in range(world)])
            out.fill(0)
            status.fill_(-1)
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), ref.ptrs(), n * E, DT[dtype], 0, stream()), "all_reduce")
            P.check(P.purlin_all_reduce_noalloc(world, src.ptrs(), out.ptrs(), n * E, DT[dtype], status, stream()),
                    "all_reduce_noalloc")
            sync()
            assert int(status.item()) == P.PL_OK, call
            for r in range(world):
                assert np.array_equal(bits(out.read(r, NP[dtype])), bits(ref.read(r, NP[dtype]))), (call, r)
            assert out.guards_intact() and src.guards_intact()
    finally:
        assert h.close() == P.PL_OK


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
    at and after the wrap all give the handle-based AllReduce's result."""
    world, n, dtype = 8, (1 << 18) + 3, "bf16"
    rng = np.random.default_rng(7)
    src = RankBuffers([n * 2] * world)
    ref = RankBuffers([n * 2] * world)
    out = RankBuffers([n * 2] * world)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda:0")
    h = Handle(world)
    try:
        P.check(P.purlin_debug_noalloc_set_epoch(0xFFFFFFFD, stream()))
        for call in range(4):
            src.upload([_draw(rng, dtype, n) for _ in range(world)])
            out.fill(0)
            status.fill_(-1)
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), ref.ptrs(), n * 2, P.PL_BF16, 0, stream()))
            P.check(P.purlin_all_reduce_noalloc(world, src.ptrs(), out.ptrs(), n * 2, P.PL_BF16, status, stream()))
            sync()
            assert int(status.item()) == P.PL_OK, call
            for r in range(world):
                assert np.array_equal(out.read(r, np.uint16), ref.read(r, np.uint16)), (call, r)
    finally:
        assert h.close() == P.PL_OK
