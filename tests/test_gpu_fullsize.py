"""The five workloads at full size, in the launch configuration the benchmark times.

AllReduce (8 x 64 MiB bf16), ReduceScatter (8 x 256 MiB fp32 and 8 x 128 MiB
bf16), AllGather / AllToAll over the whole 1 KiB .. 256 MiB sweep, and the
V variants with counts up to 4 Mi elements.  Every output element is
compared with the oracle (the large AllGather block by block, so that the
16 GiB of outputs never sit on the host at once).
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", [P.PL_LAYOUT_AUTO, P.PL_LAYOUT_TWO_SHOT, P.PL_LAYOUT_TWO_SHOT_FUSED])
def test_allreduce_bf16_8x64MiB(layout):
    """The headline workload as the bench runs it: back-to-back launches on one
    stream (programmatic dependent launch), then every output element checked."""
    x = inputs.w2_allreduce_bf16()
    world, n = x.shape
    src = RankBuffers([n * 2] * world)
    dst = RankBuffers([n * 2] * world)
    src.upload([x[r] for r in range(world)])
    h = Handle(world)
    if layout:
        P.check(P.purlin_tune_override(h.h, {"layout": layout}))
    for _ in range(3):
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    want = oracle.all_reduce([x[r] for r in range(world)], "bf16")[0]
    for r in range(world):
        assert np.array_equal(dst.read(r, np.uint16), want), r
    assert dst.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_8x64Mi(dtype):
    x = inputs.w3_reduce_scatter(dtype=dtype)
    world, n = x.shape
    E = 4 if dtype == "f32" else 2
    src = RankBuffers([n * E] * world)
    dst = RankBuffers([n // world * E] * world)
    src.upload([x[r] for r in range(world)])
    h = Handle(world)
    P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), n * E, P.PL_F32 if dtype == "f32" else P.PL_BF16,
                                    0, stream()))
    sync()
    assert h.close() == P.PL_OK
    want = oracle.reduce_scatter([x[r] for r in range(world)], dtype)
    for r in range(world):
        assert np.array_equal(bits(dst.read(r, np.float32 if dtype == "f32" else np.uint16)), bits(want[r]))
    assert dst.guards_intact()


def test_all_gather_and_all_to_all_sweep():
    world = 8
    h = Handle(world)
    try:
        for S in inputs.W4_SIZES:
            x = inputs.w4_bytes(world, S)
            src = RankBuffers([S] * world)
            src.upload([x[r] for r in range(world)])
            # AllGather: out[r] block s == in[s]
            dst = RankBuffers([world * S] * world)
            P.check(P.purlin_all_gather(h.h, src.ptrs(), dst.ptrs(), S, stream()))
            sync()
            flat = x.reshape(-1)
            for r in range(world):
                assert np.array_equal(dst.read(r), flat), (S, r)
            assert dst.guards_intact()
            del dst
            # AllToAll
            dst = RankBuffers([S] * world)
            P.check(P.purlin_all_to_all(h.h, src.ptrs(), dst.ptrs(), S, stream()))
            sync()
            want = oracle.all_to_all([x[r] for r in range(world)])
            for r in range(world):
                assert np.array_equal(dst.read(r), want[r]), (S, r)
            assert dst.guards_intact()
            del dst, src
            torch.cuda.empty_cache()
    finally:
        assert h.close() == P.PL_OK


def test_v_variants_full_counts():
    world = 8
    C, c = inputs.w5_counts(world)
    a2av_in, agv_in = inputs.w5_payloads(C, c)
    h = Handle(world)
    try:
        src = RankBuffers([a.nbytes for a in agv_in])
        dst = RankBuffers([int(c.sum()) * 2] * world)
        src.upload(agv_in)
        P.check(P.purlin_all_gather_v(h.h, src.ptrs(), dst.ptrs(), [int(v) * 2 for v in c], stream()))
        sync()
        want = oracle.all_gather_v(agv_in, [int(v) for v in c])
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
        assert dst.guards_intact()
        src = RankBuffers([a.nbytes for a in a2av_in])
        dst = RankBuffers([int(C[:, d].sum()) * 2 for d in range(world)])
        src.upload(a2av_in)
        P.check(P.purlin_all_to_all_v(h.h, src.ptrs(), dst.ptrs(), [int(v) * 2 for v in C.reshape(-1)], stream()))
        sync()
        want = oracle.all_to_all_v(a2av_in, C)
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
        assert dst.guards_intact()
    finally:
        assert h.close() == P.PL_OK
