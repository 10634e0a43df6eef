"""Streamed bulk copies (PL_SCHED_STREAM) and the shared item queue
(PL_SCHED_QUEUE) against the oracle, byte for byte.

Cases cover every copy collective at any byte alignment of sources and
destinations, items shorter than 16 bytes (no body: head and tail only),
many items per CTA (small parts), small chunks and rings of 2..8 slots.
Each case runs twice on one handle, the destinations cleared in between: the
queue counter that the last CTA of a launch resets must start the second
launch from zero.  A CUDA graph of queued calls replays several times, and
the trace records every item exactly once.  The queue on the register path
runs every collective, the two-shot (SNAC) AllReduce included, whose
dropped-notify time-out must leave the next calls correct.
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

RNG = np.random.default_rng(77)
FN = {"ag": P.purlin_all_gather, "a2a": P.purlin_all_to_all, "agv": P.purlin_all_gather_v,
      "a2av": P.purlin_all_to_all_v}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


def run_twice(kind, world, ins, sizes_arg, out_sizes, tune, smis=None, dmis=None):
    src = RankBuffers([a.nbytes for a in ins], smis)
    dst = RankBuffers(out_sizes, dmis)
    src.upload(ins)
    h = Handle(world)
    outs = []
    try:
        P.check(P.purlin_tune_override(h.h, tune))
        for _ in range(2):
            dst.fill(0)
            P.check(FN[kind](h.h, src.ptrs(), dst.ptrs(), sizes_arg, stream()), kind)
            sync()
            assert h.status() == 0
            assert dst.guards_intact()
            outs.append([dst.read(r) for r in range(world)])
    finally:
        assert h.close() == P.PL_OK
    return outs


def expect(outs, want, view=None):
    for call in outs:
        for r, w in enumerate(want):
            got = call[r] if view is None else call[r].view(view)
            assert np.array_equal(got, w), r


SCHED = [P.PL_SCHED_STREAM, P.PL_SCHED_QUEUE, P.PL_SCHED_QUEUE_GUIDED]


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("stages,chunk", [(2, 4096), (3, 8192), (8, 2048)])
def test_stream_all_gather_and_all_to_all(schedule, stages, chunk):
    tune = {"path": P.PATH_BULK, "schedule": schedule, "stages": stages, "chunk_bytes": chunk,
            "interleave_bytes": 8192}
    world = 8
    for S in (8, 16, 4096 + 8, 65536 + 48, (1 << 20) + 16 * 8):
        ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        expect(run_twice("ag", world, ins, S, [world * S] * world, tune), oracle.all_gather(ins))
        expect(run_twice("a2a", world, ins, S, [S] * world, tune), oracle.all_to_all(ins))


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("smis,dmis", [([1, 3, 5, 7], [0, 0, 0, 0]), ([0, 0, 0, 0], [9, 2, 15, 4]),
                                       ([3, 11, 6, 1], [14, 5, 0, 8]), ([2, 6, 10, 14], [2, 2, 2, 2])])
def test_stream_copies_at_any_byte_alignment(schedule, smis, dmis):
    tune = {"path": P.PATH_BULK, "schedule": schedule, "stages": 3, "chunk_bytes": 4096,
            "interleave_bytes": 4096}
    world = 4
    for S in (4, 33, 1003, 100001 * 4):
        ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        expect(run_twice("ag", world, ins, S, [world * S] * world, tune, smis, dmis), oracle.all_gather(ins))
        S2 = S - S % world
        ins2 = [x[:S2].copy() for x in ins]
        expect(run_twice("a2a", world, ins2, S2, [S2] * world, tune, smis, dmis), oracle.all_to_all(ins2))


@pytest.mark.parametrize("schedule", SCHED)
@pytest.mark.parametrize("world", [2, 3, 8])
def test_stream_v_variants(schedule, world):
    tune = {"path": P.PATH_BULK, "schedule": schedule, "stages": 4, "chunk_bytes": 8192}
    C, c = inputs.w5_counts(world, max_count=30000, seed=4)
    a2av_in, agv_in = inputs.w5_payloads(C, c, seed=4)
    outs = run_twice("agv", world, agv_in, [int(v) * 2 for v in c], [int(c.sum()) * 2] * world, tune)
    expect(outs, oracle.all_gather_v(agv_in, [int(v) for v in c]), np.uint16)
    outs = run_twice("a2av", world, a2av_in, [int(v) * 2 for v in C.reshape(-1)],
                     [int(C[:, d].sum()) * 2 for d in range(world)], tune)
    expect(outs, oracle.all_to_all_v(a2av_in, C), np.uint16)


@pytest.mark.parametrize("schedule", SCHED)
def test_stream_atom_copy(schedule):
    h = Handle(1)
    try:
        P.check(P.purlin_tune_override(h.h, {"path": P.PATH_BULK, "schedule": schedule, "stages": 3,
                                             "chunk_bytes": 16384, "interleave_bytes": 65536}))
        for S, sm, dm in ((7, 0, 0), (1 << 20, 0, 0), ((3 << 20) + 5, 3, 0), ((1 << 20) + 2, 0, 6)):
            x = RNG.integers(0, 256, size=S, dtype=np.uint8)
            src = RankBuffers([S], [sm])
            dst = RankBuffers([S] * 3, [dm] * 3)
            src.upload([x])
            for _ in range(2):
                dst.fill(0)
                P.check(P.purlin_atom_copy(h.h, src.ptr(0), dst.ptrs(), S, stream()))
                sync()
                assert dst.guards_intact()
                for r in range(3):
                    assert np.array_equal(dst.read(r), x), (S, r)
    finally:
        assert h.close() == P.PL_OK


def test_queue_in_a_cuda_graph():
    world = 8
    C, _ = inputs.w5_counts(world, max_count=40000, seed=9)
    a2av_in, _ = inputs.w5_payloads(C, np.zeros(world, np.int64), seed=9)
    src = RankBuffers([a.nbytes for a in a2av_in])
    dst = RankBuffers([int(C[:, d].sum()) * 2 for d in range(world)])
    src.upload(a2av_in)
    sizes = [int(v) * 2 for v in C.reshape(-1)]
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, {"path": P.PATH_BULK, "schedule": P.PL_SCHED_QUEUE,
                                             "interleave_bytes": 16384}))
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            P.check(P.purlin_all_to_all_v(h.h, src.ptrs(), dst.ptrs(), sizes, s.cuda_stream))  # builds the plan
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(3):
                    P.check(P.purlin_all_to_all_v(h.h, src.ptrs(), dst.ptrs(), sizes, s.cuda_stream))
            want = oracle.all_to_all_v(a2av_in, C)
            for _ in range(4):
                dst.fill(0)
                g.replay()
                s.synchronize()
                for r in range(world):
                    assert np.array_equal(dst.read(r).view(np.uint16), want[r])
            del g
        assert h.status() == 0
    finally:
        assert h.close() == P.PL_OK


@pytest.mark.parametrize("schedule", SCHED)
def test_stream_trace_records_every_item(schedule):
    world, S = 4, 300000 + 4
    ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
    tune = {"path": P.PATH_BULK, "schedule": schedule, "stages": 3, "chunk_bytes": 4096,
            "interleave_bytes": 8192}
    src = RankBuffers([S] * world, [1, 0, 3, 0])
    dst = RankBuffers([S] * world, [0, 5, 0, 2])
    src.upload(ins)
    st, items, grid, _ = P.purlin_plan_describe(P.PL_COLL_ALL_TO_ALL, world, P.PL_U8, [S], src.ptrs(), dst.ptrs(),
                                                torch.cuda.get_device_properties(0).multi_processor_count, tune)
    assert st == P.PL_OK
    cap = len(items) + 16
    buf = torch.zeros(8 + 32 * cap, dtype=torch.uint8, device="cuda:0")
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, tune))
        P.check(P.purlin_trace_enable(h.h, buf, buf.numel()))
        P.check(P.purlin_all_to_all(h.h, src.ptrs(), dst.ptrs(), S, stream()))
        sync()
        P.check(P.purlin_trace_enable(h.h, None, 0))
    finally:
        assert h.close() == P.PL_OK
    count, recs = P.trace_records(buf.cpu().numpy().tobytes())
    assert count == len(items)
    assert sorted(r["item"] for r in recs) == list(range(len(items)))
    for r in recs:
        assert r["end_ns"] >= r["start_ns"] and r["cta"] < grid
        if schedule == P.PL_SCHED_STREAM:
            assert r["cta"] == items[r["item"]]["cta"]
    want = oracle.all_to_all(ins)
    for r in range(world):
        assert np.array_equal(dst.read(r), want[r])


# ------------------------------------------- the shared queue on the register path

REGQ = {"path": P.PATH_REGISTER, "schedule": P.PL_SCHED_QUEUE}


def draw(dtype, n):
    x = RNG.standard_normal(n).astype(np.float32)
    return x if dtype == "f32" else inputs.to_bf16_bits(x)


@pytest.mark.parametrize("layout", [P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("world", [2, 5, 8])
def test_queued_all_reduce(layout, dtype, world):
    E = 4 if dtype == "f32" else 2
    n = 70001 * world + 3
    ins = [draw(dtype, n) for _ in range(world)]
    src = RankBuffers([n * E] * world, [0, 4, 8, 12, 0, 4, 8, 12][:world] if dtype == "f32" else None)
    dst = RankBuffers([n * E] * world)
    src.upload(ins)
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, dict(REGQ, layout=layout, chunk_bytes=8192, interleave_bytes=16384)))
        want = oracle.all_reduce(ins, dtype)
        for _ in range(2):
            dst.fill(0)
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * E, P.PL_F32 if dtype == "f32" else P.PL_BF16,
                                        0, stream()))
            sync()
            assert h.status() == 0
            for r in range(world):
                got = dst.read(r, np.float32 if dtype == "f32" else np.uint16)
                assert np.array_equal(got.view(np.uint32) if dtype == "f32" else got,
                                      want[r].view(np.uint32) if dtype == "f32" else want[r]), r
        assert dst.guards_intact()
    finally:
        assert h.close() == P.PL_OK


def test_queued_register_copies_and_reduce_scatter():
    world = 8
    tune = dict(REGQ, interleave_bytes=8192)
    for S in (8 * 1000 + 8, 65536 + 48, (1 << 20) + 16 * 8):
        ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        expect(run_twice("ag", world, ins, S, [world * S] * world, tune, [1, 0, 3, 0, 5, 0, 7, 0]),
               oracle.all_gather(ins))
        expect(run_twice("a2a", world, ins, S, [S] * world, tune), oracle.all_to_all(ins))
    C, c = inputs.w5_counts(world, max_count=30000, seed=4)
    a2av_in, agv_in = inputs.w5_payloads(C, c, seed=4)
    expect(run_twice("agv", world, agv_in, [int(v) * 2 for v in c], [int(c.sum()) * 2] * world, tune),
           oracle.all_gather_v(agv_in, [int(v) for v in c]), np.uint16)
    expect(run_twice("a2av", world, a2av_in, [int(v) * 2 for v in C.reshape(-1)],
                     [int(C[:, d].sum()) * 2 for d in range(world)], tune), oracle.all_to_all_v(a2av_in, C), np.uint16)
    n = 8 * 50001
    ins = [draw("f32", n) for _ in range(world)]
    src = RankBuffers([n * 4] * world)
    dst = RankBuffers([n // world * 4] * world)
    src.upload(ins)
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, tune))
        want = oracle.reduce_scatter(ins, "f32")
        for _ in range(2):
            dst.fill(0)
            P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
            sync()
            for r in range(world):
                assert np.array_equal(dst.read(r, np.float32).view(np.uint32), want[r].view(np.uint32))
    finally:
        assert h.close() == P.PL_OK


def test_queued_two_shot_wait_runs_out_and_recovers():
    world, n = 4, 1 << 16
    ins = [draw("f32", n) for _ in range(world)]
    src = RankBuffers([n * 4] * world)
    dst = RankBuffers([n * 4] * world)
    src.upload(ins)
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, dict(REGQ, layout=P.PL_LAYOUT_TWO_SHOT, chunk_bytes=4096)))
        P.check(P.purlin_set_wait_timeout_ns(h.h, 20_000_000))
        P.check(P.purlin_debug_drop_notify(h.h, 0))          # item 0 is a reduce that notifies
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
        sync()
        assert h.status() == P.PL_ERR_TIMEOUT
        assert h.status() == 0
        want = oracle.all_reduce(ins, "f32")
        for _ in range(2):                                   # the queue counter starts from zero again
            dst.fill(0)
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
            sync()
            assert h.status() == 0
            for r in range(world):
                assert np.array_equal(dst.read(r, np.float32).view(np.uint32), want[r].view(np.uint32))
    finally:
        assert h.close() == P.PL_OK


def test_queued_two_shot_in_a_cuda_graph():
    world, n = 8, (1 << 18) + 5
    ins = [draw("bf16", n) for _ in range(world)]
    src = RankBuffers([n * 2] * world)
    dst = RankBuffers([n * 2] * world)
    src.upload(ins)
    h = Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, dict(REGQ, layout=P.PL_LAYOUT_TWO_SHOT, chunk_bytes=16384)))
        s = torch.cuda.Stream()
        want = oracle.all_reduce(ins, "bf16")
        with torch.cuda.stream(s):
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, s.cuda_stream))
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(3):
                    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, s.cuda_stream))
            for _ in range(3):
                dst.fill(0)
                g.replay()
                s.synchronize()
                for r in range(world):
                    assert np.array_equal(dst.read(r, np.uint16), want[r])
            del g
        assert h.status() == 0
    finally:
        assert h.close() == P.PL_OK


@pytest.mark.parametrize("schedule", SCHED)
def test_stream_sixteen_ranks(schedule):
    """Sixteen destinations per AllGather item (every pointer slot of an item)."""
    tune = {"path": P.PATH_BULK, "schedule": schedule, "stages": 3, "chunk_bytes": 8192, "interleave_bytes": 8192}
    world = 16
    for S in (48, 65536 + 16 * 3):
        ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        expect(run_twice("ag", world, ins, S, [world * S] * world, tune, [r % 16 for r in range(world)]),
               oracle.all_gather(ins))
        expect(run_twice("a2a", world, ins, S, [S] * world, tune), oracle.all_to_all(ins))
