"""The ring AllReduce layout on the GPU, against the ring oracle.

Chunk j's partial sum starts at rank j and gains one rank per hop, each hop a
reduce item of two sources (the rank's input and the partial the previous
hop stored in the previous rank's output) that waits for the previous hop's
flag; then the finished chunks are copied around the ring.  The results must
equal oracle.all_reduce_ring bit for bit: over worlds 2..16, both dtypes,
ragged sizes, unaligned buffers, in place, repeated calls and CUDA-graph
replays on one handle, the register queue, a caller workspace sized by
purlin_workspace_bytes, and the full 8 x 64 MiB bf16 workload.  For three or
more ranks the ring's results differ from the ascending fold, so the tests
tell the two apart.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_datapath_reduce_gb300 import _build, inputs
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle, RankBuffers, stream, sync

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(2024)
ESZ = {"f32": 4, "bf16": 2}
DT = {"f32": P.PL_F32, "bf16": P.PL_BF16}
NP = {"f32": np.float32, "bf16": np.uint16}
RING = {"layout": P.PL_LAYOUT_RING}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


def draw(dtype, n):
    x = RNG.standard_normal(n).astype(np.float32)
    return x if dtype == "f32" else inputs.to_bf16_bits(x)


def bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def run_ring(world, dtype, n, tune=None, misalign=None, ins=None, h=None):
    E = ESZ[dtype]
    ins = ins if ins is not None else [draw(dtype, n) for _ in range(world)]
    src = RankBuffers([n * E] * world, misalign)
    dst = RankBuffers([n * E] * world, misalign)
    src.upload(ins)
    own = h is None
    h = h or Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, dict(RING, **(tune or {}))))
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * E, DT[dtype], 0, stream()), "ring")
        sync()
        assert h.status() == 0
    finally:
        if own:
            assert h.close() == P.PL_OK
    assert dst.guards_intact() and src.guards_intact()
    return ins, [dst.read(r, NP[dtype]) for r in range(world)]


@pytest.mark.parametrize("world", [2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ring_matches_oracle(world, dtype):
    for n in (1, 3, 8, 1000, 4099, 65536 + 7, (1 << 20) + 5):
        ins, outs = run_ring(world, dtype, n, tune={"chunk_bytes": 16384})
        want = oracle.all_reduce_ring(ins, dtype)
        for r in range(world):
            assert np.array_equal(bits(outs[r]), bits(want[r])), (n, r)


def test_ring_differs_from_ascending_fold():
    """Three or more ranks: some sums differ from the ascending fold (the
    kernel really folds in ring order); two ranks: identical."""
    ins, outs = run_ring(8, "bf16", 1 << 16)
    ring, asc = oracle.all_reduce_ring(ins, "bf16"), oracle.all_reduce(ins, "bf16")
    assert np.array_equal(outs[0], ring[0]) and not np.array_equal(outs[0], asc[0])
    ins, outs = run_ring(2, "f32", 4099)
    assert np.array_equal(bits(outs[1]), bits(oracle.all_reduce(ins, "f32")[1]))
    # the hand-worked order case: chunk j folded from rank j
    x = [np.array([v] * 3, dtype=np.float32) for v in (1e8, 1.0, -1e8)]
    _, outs = run_ring(3, "f32", 3, ins=x)
    assert [list(o) for o in outs] == [[0.0, 0.0, 1.0]] * 3


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ring_unaligned_buffers(dtype):
    E = ESZ[dtype]
    for misalign in ([E, 2 * E, 0, 3 * E], [4 * E, 0, 12 // E * E, 8]):
        misalign = [m - m % E for m in misalign]
        ins, outs = run_ring(4, dtype, 50001, misalign=misalign, tune={"chunk_bytes": 8192})
        want = oracle.all_reduce_ring(ins, dtype)
        for r in range(4):
            assert np.array_equal(bits(outs[r]), bits(want[r]))


def test_ring_in_place():
    world, n, dtype = 8, 300007, "bf16"
    ins = [draw(dtype, n) for _ in range(world)]
    buf = RankBuffers([n * 2] * world)
    buf.upload(ins)
    h = Handle(world)
    P.check(P.purlin_tune_override(h.h, dict(RING, chunk_bytes=8192)))
    P.check(P.purlin_all_reduce(h.h, buf.ptrs(), buf.ptrs(), n * 2, P.PL_BF16, 0, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    want = oracle.all_reduce_ring(ins, dtype)
    for r in range(world):
        assert np.array_equal(buf.read(r, np.uint16), want[r])
    assert buf.guards_intact()


def test_ring_repeated_calls_and_graph_replays():
    """Epochs advance from call to call; a captured call replays correctly."""
    world, n = 8, (1 << 18) + 3
    h = Handle(world)
    try:
        for _ in range(3):
            ins, outs = run_ring(world, "bf16", n, tune={"chunk_bytes": 16384}, h=h)
            want = oracle.all_reduce_ring(ins, "bf16")
            for r in range(world):
                assert np.array_equal(outs[r], want[r])
        ins = [draw("bf16", n) for _ in range(world)]
        src = RankBuffers([n * 2] * world)
        dst = RankBuffers([n * 2] * world)
        src.upload(ins)
        s = torch.cuda.Stream()
        call = lambda: P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, s.cuda_stream))
        with torch.cuda.stream(s):
            call()                      # builds the plan before capture
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(3):
                    call()
            dst.fill(0)
            for _ in range(2):
                g.replay()
            s.synchronize()
        st, dv = P.purlin_status_get(h.h, s.cuda_stream)
        assert st == 0 and dv == 0
        want = oracle.all_reduce_ring(ins, "bf16")
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK


def test_ring_on_the_register_queue():
    for world in (3, 8):
        ins, outs = run_ring(world, "f32", 200003, tune={"chunk_bytes": 4096, "schedule": P.PL_SCHED_QUEUE})
        want = oracle.all_reduce_ring(ins, "f32")
        for r in range(world):
            assert np.array_equal(bits(outs[r]), bits(want[r]))


def test_ring_in_caller_workspace():
    """A workspace of purlin_workspace_bytes(world, S) holds the ring's flags at the table's tile size."""
    world, S = 8, 16 << 20
    nb = P.purlin_workspace_bytes(world, S)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda:0")
    h = Handle(world, ws.data_ptr(), nb)
    try:
        ins, outs = run_ring(world, "bf16", S // 2, h=h)
        want = oracle.all_reduce_ring(ins, "bf16")
        for r in range(world):
            assert np.array_equal(outs[r], want[r])
    finally:
        assert h.close() == P.PL_OK


def test_ring_full_workload_8x64MiB():
    """The bench's ring workload: 8 ranks x 32 Mi bf16 elements, every output element checked."""
    world, n = 8, 32 << 20
    x = inputs.w2_allreduce_bf16(world, n, seed=1)
    ins = [x[r] for r in range(world)]
    _, outs = run_ring(world, "bf16", n, ins=ins)
    want = oracle.all_reduce_ring(ins, "bf16")
    for r in range(world):
        assert np.array_equal(outs[r], want[r]), r
    torch.cuda.empty_cache()
