"""The library-owned workspace: sized at initialize, grown only past its stated capacity.

A handle created without a caller's workspace holds the SNAC flags of the
two-shot and ring layouts up to the sizes the header states, so their first
calls at the workload sizes do not grow it (no allocation, no device-wide
synchronisation inside a collective).  A call past that capacity grows it
once, between launches, and its results are still the oracle's.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


def _run(h, world, ins, tune):
    n = ins[0].size
    src = RankBuffers([n * 2] * world)
    dst = RankBuffers([n * 2] * world)
    src.upload(ins)
    P.check(P.purlin_tune_override(h.h, tune))
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
    sync()
    assert h.status() == 0
    outs = [dst.read(r, np.uint16) for r in range(world)]
    assert dst.guards_intact() and src.guards_intact()
    return outs


def test_snac_layouts_at_the_workload_size_do_not_grow_it():
    world, n = 8, 32 << 20
    x = inputs.w2_allreduce_bf16(world, n, seed=1)
    ins = [x[r] for r in range(world)]
    want = oracle.all_reduce(ins, "bf16")
    h = Handle(world)
    try:
        st, nbytes, grown = P.purlin_workspace_query(h.h)
        assert st == P.PL_OK and grown == 0 and nbytes >= 256 + 4 * (2 << 20)
        for layout in (P.PL_LAYOUT_TWO_SHOT, P.PL_LAYOUT_RING):
            outs = _run(h, world, ins, {"layout": layout})
            for r in range(world):
                assert np.array_equal(outs[r], want[r]), (layout, r)
        assert P.purlin_workspace_query(h.h)[2] == 0
    finally:
        assert h.close() == P.PL_OK
    torch.cuda.empty_cache()


def test_initialize_takes_a_size_for_its_own_workspace():
    """workspace NULL with workspace_bytes above the default: the library allocates that much."""
    big = P.purlin_workspace_bytes(16, 8 << 30)
    h = Handle(16, None, big)
    try:
        st, nbytes, grown = P.purlin_workspace_query(h.h)
        assert st == P.PL_OK and nbytes == big and grown == 0
    finally:
        assert h.close() == P.PL_OK


def test_past_the_capacity_it_grows_once_and_stays_exact():
    """16 ranks x 80 MiB, ring tiles of 1 KiB: about 2.4 million flags, more
    than the default 2 Mi; the call grows the workspace once."""
    world, n = 16, 40 << 20
    rng = np.random.default_rng(17)
    ins = [inputs.to_bf16_bits(rng.standard_normal(n).astype(np.float32)) for _ in range(world)]
    h = Handle(world)
    try:
        outs = _run(h, world, ins, {"layout": P.PL_LAYOUT_RING, "chunk_bytes": 1024})
        assert P.purlin_workspace_query(h.h)[2] == 1
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(outs[r], want[r]), r
        outs = _run(h, world, ins, {"layout": P.PL_LAYOUT_RING, "chunk_bytes": 1024})
        assert P.purlin_workspace_query(h.h)[2] == 1         # no second growth
        for r in range(world):
            assert np.array_equal(outs[r], want[r]), r
    finally:
        assert h.close() == P.PL_OK
    torch.cuda.empty_cache()
