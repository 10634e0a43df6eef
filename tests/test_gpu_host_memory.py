"""Rank buffers in host memory: the kernel reads and writes them in place.

Pinned host buffers (torch pin_memory, i.e. cudaHostAlloc), host memory
registered after allocation (cudaHostRegister on a numpy array), a mix of
host and device ranks, in-place AllReduce on host memory, and sizes at which
device buffers would take the bulk engines (host-memory calls must run on
the register path).  Outputs equal the oracle bit for bit.  Unregistered
pageable memory is refused with PL_ERR_INVALID_ARG before anything is
launched.
"""

import numpy as np
import pytest
import torch

import oracle
import workload_inputs as inputs
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle, stream, sync

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(515)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


def pinned(a):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1).copy())
    return t.pin_memory()


def pinned_empty(nbytes):
    return torch.empty(nbytes, dtype=torch.uint8).pin_memory()


def test_all_reduce_on_pinned_host_buffers():
    world, n = 8, (1 << 19) + 3
    ins = [inputs.to_bf16_bits(RNG.standard_normal(n).astype(np.float32)) for _ in range(world)]
    src = [pinned(x) for x in ins]
    dst = [pinned_empty(n * 2) for _ in range(world)]
    h = Handle(world)
    try:
        for _ in range(2):
            P.check(P.purlin_all_reduce(h.h, src, dst, n * 2, P.PL_BF16, 0, stream()))
            sync()
            assert h.status() == 0
            want = oracle.all_reduce(ins, "bf16")
            for r in range(world):
                assert np.array_equal(dst[r].numpy().view(np.uint16), want[r])
        # in place on host memory
        P.check(P.purlin_all_reduce(h.h, src, src, n * 2, P.PL_BF16, 0, stream()))
        sync()
        for r in range(world):
            assert np.array_equal(src[r].numpy().view(np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK


def test_bulk_sized_calls_on_host_memory():
    """Sizes whose device-memory plans use the bulk engines."""
    world = 8
    h = Handle(world)
    try:
        n = (16 << 20) // 4                                   # ReduceScatter fp32, 16 MiB per rank
        ins = [RNG.standard_normal(n).astype(np.float32) for _ in range(world)]
        src = [pinned(x) for x in ins]
        dst = [pinned_empty(n // world * 4) for _ in range(world)]
        P.check(P.purlin_reduce_scatter(h.h, src, dst, n * 4, P.PL_F32, 0, stream()))
        sync()
        want = oracle.reduce_scatter(ins, "f32")
        for r in range(world):
            assert np.array_equal(dst[r].numpy().view(np.uint32), want[r].view(np.uint32))
        S = (32 << 20) + 16 * world                            # AllToAll, host sources, device destinations
        xs = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        src = [pinned(x) for x in xs]
        dst = [torch.empty(S, dtype=torch.uint8, device="cuda:0") for _ in range(world)]
        P.check(P.purlin_all_to_all(h.h, src, dst, S, stream()))
        sync()
        want = oracle.all_to_all(xs)
        for r in range(world):
            assert np.array_equal(dst[r].cpu().numpy(), want[r])
        S = (16 << 20) + 5                                     # AllGather, device sources, host destinations
        xs = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        src = [torch.from_numpy(x).to("cuda:0") for x in xs]
        dst = [pinned_empty(world * S) for _ in range(world)]
        P.check(P.purlin_all_gather(h.h, src, dst, S, stream()))
        sync()
        flat = np.concatenate(xs)
        for r in range(world):
            assert np.array_equal(dst[r].numpy(), flat)
        assert h.status() == 0
    finally:
        assert h.close() == P.PL_OK


def test_v_variants_on_host_memory():
    world = 8
    C, c = inputs.w5_counts(world, max_count=300000, seed=4)
    a2av_in, agv_in = inputs.w5_payloads(C, c, seed=4)
    h = Handle(world)
    try:
        src = [pinned(a) if a.size else None for a in agv_in]
        dst = [pinned_empty(int(c.sum()) * 2) for _ in range(world)]
        P.check(P.purlin_all_gather_v(h.h, src, dst, [int(v) * 2 for v in c], stream()))
        sync()
        want = oracle.all_gather_v(agv_in, [int(v) for v in c])
        for r in range(world):
            assert np.array_equal(dst[r].numpy().view(np.uint16), want[r])
        src = [pinned(a) if a.size else None for a in a2av_in]
        dst = [pinned_empty(max(1, int(C[:, d].sum()) * 2)) for d in range(world)]
        P.check(P.purlin_all_to_all_v(h.h, src, dst, [int(v) * 2 for v in C.reshape(-1)], stream()))
        sync()
        want = oracle.all_to_all_v(a2av_in, C)
        for d in range(world):
            assert np.array_equal(dst[d].numpy()[:int(C[:, d].sum()) * 2].view(np.uint16), want[d])
    finally:
        assert h.close() == P.PL_OK


def page_aligned(n, fill=None, draw=False):
    """n float32 in whole pages of their own (for cudaHostRegister)."""
    pages = (n * 4 + 4095) // 4096 + 1
    raw = np.empty(pages * 4096, np.uint8)
    off = (-raw.ctypes.data) % 4096
    a = raw[off:off + (pages - 1) * 4096].view(np.float32)[:n]
    a[:] = RNG.standard_normal(n).astype(np.float32) if draw else fill   # pages touched
    return a


def test_registered_and_pageable_host_memory():
    world, n = 4, 100003
    ins = [page_aligned(n, draw=True) for _ in range(world)]
    outs = [page_aligned(n, -1.0) for _ in range(world)]
    rt = torch.cuda.cudart()
    want = oracle.all_reduce(ins, "f32")
    h = Handle(world)
    try:
        # unregistered pageable memory is refused before anything is launched
        st = P.purlin_all_reduce(h.h, [x.ctypes.data for x in ins], [y.ctypes.data for y in outs], n * 4,
                                 P.PL_F32, 0, stream())
        assert st == P.PL_ERR_INVALID_ARG
        assert all(np.all(y == -1.0) for y in outs)
        # the same arrays registered with the driver
        for a in ins + outs:
            assert int(rt.cudaHostRegister(a.ctypes.data, (a.nbytes + 4095) // 4096 * 4096, 0)) == 0
        try:
            P.check(P.purlin_all_reduce(h.h, [x.ctypes.data for x in ins], [y.ctypes.data for y in outs], n * 4,
                                        P.PL_F32, 0, stream()))
            sync()
            for r in range(world):
                assert np.array_equal(outs[r].view(np.uint32), want[r].view(np.uint32))
        finally:
            for a in ins + outs:
                rt.cudaHostUnregister(a.ctypes.data)
        assert h.status() == 0
    finally:
        assert h.close() == P.PL_OK


def test_two_shot_on_pinned_host_buffers():
    """SNAC across CTAs with the data in host memory: reduce into the owner's
    host buffer, notify, then copies read it back from host memory."""
    world, n = 8, (1 << 18) + 5
    ins = [inputs.to_bf16_bits(RNG.standard_normal(n).astype(np.float32)) for _ in range(world)]
    src = [pinned(x) for x in ins]
    dst = [pinned_empty(n * 2) for _ in range(world)]
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 16384}))
        want = oracle.all_reduce(ins, "bf16")
        for _ in range(2):
            P.check(P.purlin_all_reduce(h.h, src, dst, n * 2, P.PL_BF16, 0, stream()))
            sync()
            assert h.status() == 0
            for r in range(world):
                assert np.array_equal(dst[r].numpy().view(np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK


def test_ring_on_pinned_host_buffers():
    """The ring's running sums live in host memory between stages (loads through the L2)."""
    world, n = 4, (1 << 17) + 3
    ins = [inputs.to_bf16_bits(RNG.standard_normal(n).astype(np.float32)) for _ in range(world)]
    src = [pinned(x) for x in ins]
    dst = [pinned_empty(n * 2) for _ in range(world)]
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, {"layout": P.PL_LAYOUT_RING, "chunk_bytes": 16384}))
        want = oracle.all_reduce(ins, "bf16")
        for _ in range(2):
            P.check(P.purlin_all_reduce(h.h, src, dst, n * 2, P.PL_BF16, 0, stream()))
            sync()
            assert h.status() == 0
            for r in range(world):
                assert np.array_equal(dst[r].numpy().view(np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK
