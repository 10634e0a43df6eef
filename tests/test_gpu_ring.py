"""The ring AllReduce layout on the GPU, against the oracle's ascending fold.

Per tile, stage k adds rank k's input to the running binary32 sum the
previous stage left in the outputs (bf16: two 16-bit halves in two ranks'
outputs), each stage waiting for the previous one's flag; then the finished
tile is passed around the ring.  Every tile is walked from rank 0 upwards, so
the results must equal oracle.all_reduce bit for bit -- max-ulp 0, inside the
1-ulp bound any reordered variant must meet -- over worlds 2..16, both
dtypes, ragged sizes, unaligned buffers, in place, repeated calls and
CUDA-graph replays on one handle, the register queue, a caller workspace
sized by purlin_workspace_bytes, and the full 8 x 64 MiB bf16 workload.
"""

import numpy as np
import pytest
import torch

import oracle
import workload_inputs as inputs
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle, RankBuffers, stream, sync
from ulp import max_ulp

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
        want = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert max_ulp(outs[r], want[r]) == 0, (n, r)
            assert np.array_equal(bits(outs[r]), bits(want[r])), (n, r)


def test_ring_folds_in_ascending_rank_order():
    """Inputs whose binary32 sum depends on the order of the adds: ranks
    [1e8, 1, -1e8] fold to (1e8 + 1) - 1e8 = 0 (1e8 + 1 rounds to 1e8), and
    [1e8, -1e8, 1] to 1, for every element whatever chunk or tile it is in.
    bf16 ranks [1, 2^-8, 2^-8]: the binary32 sum 1 + 2^-7 is exact and is
    rounded once, to 0x3F81; rounding the running sum at every stage would
    give 1.0 (0x3F80)."""
    for vals, want in (((1e8, 1.0, -1e8), 0.0), ((1e8, -1e8, 1.0), 1.0)):
        x = [np.full(5, v, dtype=np.float32) for v in vals]
        _, outs = run_ring(3, "f32", 5, ins=x)
        assert all(list(o) == [want] * 5 for o in outs), outs
    b = [np.full(9, h, dtype=np.uint16) for h in (0x3F80, 0x3B80, 0x3B80)]
    _, outs = run_ring(3, "bf16", 9, ins=b)
    assert all(int(v) == 0x3F81 for o in outs for v in o), outs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ring_unaligned_buffers(dtype):
    E = ESZ[dtype]
    for misalign in ([E, 2 * E, 0, 3 * E], [4 * E, 0, 12 // E * E, 8]):
        misalign = [m - m % E for m in misalign]
        ins, outs = run_ring(4, dtype, 50001, misalign=misalign, tune={"chunk_bytes": 8192})
        want = oracle.all_reduce(ins, dtype)
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
    want = oracle.all_reduce(ins, dtype)
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
            want = oracle.all_reduce(ins, "bf16")
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
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK


def test_ring_on_the_register_queue():
    for world in (3, 8):
        ins, outs = run_ring(world, "f32", 200003, tune={"chunk_bytes": 4096, "schedule": P.PL_SCHED_QUEUE})
        want = oracle.all_reduce(ins, "f32")
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
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(outs[r], want[r])
    finally:
        assert h.close() == P.PL_OK


def test_ring_full_workload_8x64MiB():
    """The bench's ring workload: 8 ranks x 32 Mi bf16 elements, every output
    element checked; the max-ulp distance to the ascending fold is 0."""
    world, n = 8, 32 << 20
    x = inputs.w2_allreduce_bf16(world, n, seed=1)
    ins = [x[r] for r in range(world)]
    _, outs = run_ring(world, "bf16", n, ins=ins)
    want = oracle.all_reduce(ins, "bf16")
    for r in range(world):
        assert max_ulp(outs[r], want[r]) == 0, r
        assert np.array_equal(outs[r], want[r]), r
    torch.cuda.empty_cache()


def test_ring_max_ulp_fp32_uniform():
    """fp32 U(-1,1) data (the ReduceScatter workload's distribution), 8 ranks:
    heavy cancellation, where a reordered fold lands far from the ascending
    one; the ring stays at max-ulp 0."""
    world, n = 8, (4 << 20) + 3
    rng = np.random.default_rng(21)
    ins = [(rng.random(n, dtype=np.float32) * np.float32(2) - np.float32(1)) for _ in range(world)]
    _, outs = run_ring(world, "f32", n, ins=ins)
    want = oracle.all_reduce(ins, "f32")
    for r in range(world):
        assert max_ulp(outs[r], want[r]) == 0, r
