"""CUDA path against the CPU oracle, element by element, through the C ABI.

Small cases span several tiles and CTAs and end on ragged tails; the full
workload sizes run in the benchmark's launch configuration.  Copies and the
ascending-rank reductions must be bit-exact.  Guard bytes around every
destination catch writes outside it.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import workload_inputs as inputs
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle, RankBuffers, bits, stream, sync

pytestmark = pytest.mark.gpu

DT = {"f32": P.PL_F32, "bf16": P.PL_BF16}
NP = {"f32": np.float32, "bf16": np.uint16}
ESZ = {"f32": 4, "bf16": 2}
RNG = np.random.default_rng(2024)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def draw(dtype, n, rng=RNG):
    x = rng.standard_normal(n).astype(np.float32)
    return x if dtype == "f32" else inputs.to_bf16_bits(x)


def run_all_reduce(world, dtype, n, layout=P.PL_LAYOUT_AUTO, misalign=None, tune=None, ins=None):
    E = ESZ[dtype]
    ins = ins if ins is not None else [draw(dtype, n) for _ in range(world)]
    src = RankBuffers([n * E] * world, misalign)
    dst = RankBuffers([n * E] * world, misalign)
    src.upload(ins)
    h = Handle(world)
    try:
        t = dict(tune or {})
        if layout:
            t["layout"] = layout
        if t:
            P.check(P.purlin_tune_override(h.h, t))
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * E, DT[dtype], 0, stream()), "all_reduce")
        sync()
        assert h.status() == 0
    finally:
        assert h.close() == P.PL_OK
    assert dst.guards_intact() and src.guards_intact()
    return ins, [dst.read(r, NP[dtype]) for r in range(world)]


# ------------------------------------------------------------- AllReduce

def test_worked_example_on_gpu():
    with open(os.path.join(os.path.dirname(__file__), "golden", "nki_allreduce_worked_example.json")) as f:
        g = json.load(f)
    for dtype in ("f32", "bf16"):
        ins = [np.asarray(x, dtype=np.float32).reshape(-1) for x in g["inputs"]]
        if dtype == "bf16":
            ins = [inputs.to_bf16_bits(x) for x in ins]
        for layout in (P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT):
            _, outs = run_all_reduce(2, dtype, 6, layout, ins=ins)
            for r in range(2):
                got = outs[r] if dtype == "f32" else oracle.bf16_bits_to_f32(outs[r])
                assert np.array_equal(got.reshape(2, 3), np.asarray(g["outputs"][r], dtype=np.float32))


def test_integer_workload_two_ranks():
    x = inputs.w1_allreduce_ints()
    for layout in (P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT):
        ins, outs = run_all_reduce(2, "f32", 1024, layout, ins=[x[0], x[1]])
        exact = x.astype(np.int64).sum(axis=0)
        for r in range(2):
            assert np.array_equal(outs[r].astype(np.int64), exact)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT])
def test_all_reduce_matches_oracle(world, dtype, layout):
    for n in (1, 3, 8, 1000, 4099, 65536 + 7, (1 << 20) + 5):
        ins, outs = run_all_reduce(world, dtype, n, layout, tune={"chunk_bytes": 16384})
        want = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert np.array_equal(bits(outs[r]), bits(want[r])), (n, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_reduce_unaligned_buffers(dtype):
    E = ESZ[dtype]
    for misalign in ([E, 2 * E, 0, 3 * E], [E] * 4, [4 * E, 0, 12 // E * E, 8]):
        misalign = [m - m % E for m in misalign]
        for layout in (P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT):
            ins, outs = run_all_reduce(4, dtype, 50001, layout, misalign=misalign)
            want = oracle.all_reduce(ins, dtype)
            for r in range(4):
                assert np.array_equal(bits(outs[r]), bits(want[r]))


@pytest.mark.parametrize("layout", [P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT])
def test_all_reduce_in_place(layout):
    world, n, dtype = 8, 300007, "bf16"
    ins = [draw(dtype, n) for _ in range(world)]
    buf = RankBuffers([n * 2] * world)
    buf.upload(ins)
    h = Handle(world)
    P.check(P.purlin_tune_override(h.h, {"layout": layout, "chunk_bytes": 8192}))
    P.check(P.purlin_all_reduce(h.h, buf.ptrs(), buf.ptrs(), n * 2, P.PL_BF16, 0, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    want = oracle.all_reduce(ins, dtype)
    for r in range(world):
        assert np.array_equal(buf.read(r, np.uint16), want[r])
    assert buf.guards_intact()


def test_signed_zero_and_subnormals():
    tiny = np.array([1, 0x80000000, 0x00000003], dtype=np.uint32).view(np.float32)
    ins = [np.tile(tiny, 100) for _ in range(3)]
    _, outs = run_all_reduce(3, "f32", 300, P.PL_LAYOUT_ONE_SHOT, ins=ins)
    want = oracle.all_reduce(ins, "f32")
    assert np.array_equal(bits(outs[0]), bits(want[0]))
    assert bits(outs[0])[1] == 0x80000000 and bits(outs[0])[0] == 3


# -------------------------------------------------------- ReduceScatter

@pytest.mark.parametrize("world", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_matches_oracle(world, dtype):
    E = ESZ[dtype]
    for chunk in (1, 7, 4099, 100003):
        n = chunk * world
        ins = [draw(dtype, n) for _ in range(world)]
        src = RankBuffers([n * E] * world)
        dst = RankBuffers([chunk * E] * world)
        src.upload(ins)
        h = Handle(world)
        P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), n * E, DT[dtype], 0, stream()))
        sync()
        assert h.close() == P.PL_OK
        want = oracle.reduce_scatter(ins, dtype)
        for r in range(world):
            assert np.array_equal(bits(dst.read(r, NP[dtype])), bits(want[r])), (chunk, r)
        assert dst.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_v(dtype):
    world, E = 8, ESZ[dtype]
    counts = [0, 1, 4099, 7, 100000, 0, 33, 65536]
    n = sum(counts)
    ins = [draw(dtype, n) for _ in range(world)]
    src = RankBuffers([n * E] * world)
    dst = RankBuffers([c * E for c in counts])
    src.upload(ins)
    h = Handle(world)
    P.check(P.purlin_reduce_scatter_v(h.h, src.ptrs(), dst.ptrs(), [c * E for c in counts], DT[dtype], 0,
                                      stream()))
    sync()
    assert h.close() == P.PL_OK
    want = oracle.reduce_scatter_v(ins, counts, dtype)
    for r in range(world):
        assert np.array_equal(bits(dst.read(r, NP[dtype])), bits(want[r]))
    assert dst.guards_intact()


# ------------------------------------------------------------------ copies

def run_copy(kind, world, ins, sizes_arg, out_sizes, smis=None, dmis=None, tune=None):
    src = RankBuffers([a.nbytes for a in ins], smis)
    dst = RankBuffers(out_sizes, dmis)
    src.upload(ins)
    dst.fill(0)
    h = Handle(world)
    if tune:
        P.check(P.purlin_tune_override(h.h, tune))
    fn = {"ag": P.purlin_all_gather, "a2a": P.purlin_all_to_all, "agv": P.purlin_all_gather_v,
          "a2av": P.purlin_all_to_all_v}[kind]
    P.check(fn(h.h, src.ptrs(), dst.ptrs(), sizes_arg, stream()), kind)
    sync()
    assert h.close() == P.PL_OK
    assert dst.guards_intact()
    return [dst.read(r) for r in range(world)]


@pytest.mark.parametrize("world", [1, 2, 3, 8, 16])
def test_all_gather_and_all_to_all(world):
    for S in (16, 1000, 4096, 65536 + 48, 1 << 20):
        S -= S % world
        ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        outs = run_copy("ag", world, ins, S, [world * S] * world)
        want = oracle.all_gather(ins)
        for r in range(world):
            assert np.array_equal(outs[r], want[r])
        outs = run_copy("a2a", world, ins, S, [S] * world)
        want = oracle.all_to_all(ins)
        for r in range(world):
            assert np.array_equal(outs[r], want[r])


def test_copies_at_any_byte_alignment():
    world = 4
    for smis, dmis in (([1, 3, 5, 7], [0, 0, 0, 0]), ([0, 0, 0, 0], [9, 2, 15, 4]), ([3, 11, 6, 1], [14, 5, 0, 8])):
        for S in (4, 33, 1003, 100001 * 4):
            ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
            outs = run_copy("ag", world, ins, S, [world * S] * world, smis, dmis)
            want = oracle.all_gather(ins)
            for r in range(world):
                assert np.array_equal(outs[r], want[r]), (smis, dmis, S)
            S2 = S - S % world
            ins2 = [x[:S2].copy() for x in ins]
            outs = run_copy("a2a", world, ins2, S2, [S2] * world, smis, dmis)
            want = oracle.all_to_all(ins2)
            for r in range(world):
                assert np.array_equal(outs[r], want[r]), (smis, dmis, S)


@pytest.mark.parametrize("world", [2, 3, 8])
def test_v_variants_with_workload_structure(world):
    C, c = inputs.w5_counts(world, max_count=5000, seed=4)
    a2av_in, agv_in = inputs.w5_payloads(C, c, seed=4)
    # AllGatherV over bf16 payload, byte counts
    outs = run_copy("agv", world, agv_in, [int(v) * 2 for v in c], [int(c.sum()) * 2] * world)
    want = oracle.all_gather_v(agv_in, [int(v) for v in c])
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])
    outs = run_copy("a2av", world, a2av_in, [int(v) * 2 for v in C.reshape(-1)],
                    [int(C[:, d].sum()) * 2 for d in range(world)])
    want = oracle.all_to_all_v(a2av_in, C)
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])


# --------------------------------------------------------------------- Atoms

def test_atom_copy_and_reduce():
    h = Handle(1)
    try:
        for nd in (1, 2, 5):
            for S in (1, 17, 4096, 300001):
                x = RNG.integers(0, 256, size=S, dtype=np.uint8)
                src = RankBuffers([S])
                dst = RankBuffers([S] * nd, [0, 1, 2, 3, 4][:nd])
                src.upload([x])
                P.check(P.purlin_atom_copy(h.h, src.ptr(0), dst.ptrs(), S, stream()))
                sync()
                for j in range(nd):
                    assert np.array_equal(dst.read(j), x)
                assert dst.guards_intact()
        for dtype in ("f32", "bf16"):
            for ns in (1, 2, 3, 8, 11):
                for nd in (1, 3):
                    n = 70001
                    xs = [draw(dtype, n) for _ in range(ns)]
                    src = RankBuffers([n * ESZ[dtype]] * ns)
                    dst = RankBuffers([n * ESZ[dtype]] * nd)
                    src.upload(xs)
                    P.check(P.purlin_atom_reduce(h.h, src.ptrs(), dst.ptrs(), n * ESZ[dtype], DT[dtype], stream()))
                    sync()
                    want = oracle.all_reduce(xs, dtype)[0]
                    for j in range(nd):
                        assert np.array_equal(bits(dst.read(j, NP[dtype])), bits(want)), (dtype, ns, nd)
    finally:
        assert h.close() == P.PL_OK


# ------------------------------------------------------ invariants on GPU

def test_repeatable_and_grid_independent():
    world, n, dtype = 8, 500003, "f32"
    ins = [draw(dtype, n) for _ in range(world)]
    ref = None
    for tune in (None, {"ctas_per_sm": 1}, {"threads": 128, "unroll": 2}, {"threads": 256, "ctas_per_sm": 4},
                 {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 4096}, {"store_hint": 2}):
        for _ in range(2):
            _, outs = run_all_reduce(world, dtype, n, tune=tune, ins=ins)
            got = np.stack([bits(o) for o in outs])
            if ref is None:
                ref = got
            assert np.array_equal(got, ref), tune


def test_all_reduce_equals_all_gather_of_reduce_scatter():
    world, chunk, dtype = 8, 40000, "bf16"
    n = world * chunk
    ins = [draw(dtype, n) for _ in range(world)]
    src = RankBuffers([n * 2] * world)
    mid = RankBuffers([chunk * 2] * world)
    ag = RankBuffers([n * 2] * world)
    ar = RankBuffers([n * 2] * world)
    src.upload(ins)
    h = Handle(world)
    P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), mid.ptrs(), n * 2, P.PL_BF16, 0, stream()))
    P.check(P.purlin_all_gather(h.h, mid.ptrs(), ag.ptrs(), chunk * 2, stream()))
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), ar.ptrs(), n * 2, P.PL_BF16, 0, stream()))
    sync()
    assert h.close() == P.PL_OK
    for r in range(world):
        assert np.array_equal(ag.read(r), ar.read(r))


def test_all_to_all_twice_is_identity():
    world, S = 8, 8 * 12345
    ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
    a = RankBuffers([S] * world)
    b = RankBuffers([S] * world)
    c = RankBuffers([S] * world)
    a.upload(ins)
    h = Handle(world)
    P.check(P.purlin_all_to_all(h.h, a.ptrs(), b.ptrs(), S, stream()))
    P.check(P.purlin_all_to_all(h.h, b.ptrs(), c.ptrs(), S, stream()))
    sync()
    assert h.close() == P.PL_OK
    for r in range(world):
        assert np.array_equal(c.read(r), ins[r])


def test_cuda_graph_replay():
    world, n = 8, 1 << 18
    ins = [draw("bf16", n) for _ in range(world)]
    src = RankBuffers([n * 2] * world)
    dst = RankBuffers([n * 2] * world)
    src.upload(ins)
    h = Handle(world)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for layout in (P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT):
            P.check(P.purlin_tune_override(h.h, {"layout": layout, "chunk_bytes": 16384}))
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, s))  # plan warm-up
            s.synchronize()
            dst.fill(0)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(3):
                    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, s))
            for _ in range(4):
                g.replay()
            s.synchronize()
            want = oracle.all_reduce(ins, "bf16")
            for r in range(world):
                assert np.array_equal(dst.read(r, np.uint16), want[r]), layout
    assert h.status() == 0
    assert h.close() == P.PL_OK


# ----------------------------------------------------------- error paths

def test_argument_errors():
    world, n = 4, 1024
    src = RankBuffers([n * 4] * world)
    dst = RankBuffers([n * 4] * world)
    h = Handle(world)
    S = stream()
    overlapping = [dst.ptr(0)] * world
    assert P.purlin_all_reduce(h.h, src.ptrs(), overlapping, n * 4, P.PL_F32, 0, S) == P.PL_ERR_INVALID_ARG
    bad = [p + 2 for p in src.ptrs()]
    assert P.purlin_all_reduce(h.h, bad, dst.ptrs(), 64, P.PL_F32, 0, S) == P.PL_ERR_ALIGNMENT
    assert P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), 64, P.PL_U8, 0, S) == P.PL_ERR_UNSUPPORTED
    assert P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), 64, P.PL_F32, 5, S) == P.PL_ERR_UNSUPPORTED
    assert P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), 12, P.PL_F32, 0, S) == P.PL_ERR_INVALID_ARG
    assert P.purlin_all_to_all(h.h, src.ptrs(), dst.ptrs(), 10, S) == P.PL_ERR_INVALID_ARG
    assert P.purlin_all_reduce(h.h, [0] * world, dst.ptrs(), 64, P.PL_F32, 0, S) == P.PL_ERR_INVALID_ARG
    # an address the driver does not know is refused before any launch
    assert P.purlin_all_reduce(h.h, [0x10000 * (r + 1) for r in range(world)], dst.ptrs(), 64, P.PL_F32, 0,
                               S) == P.PL_ERR_INVALID_ARG
    assert P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), 0, P.PL_F32, 0, S) == P.PL_OK  # zero bytes: no launch
    # sizes whose totals or buffer ends do not fit in 64 bits are refused before any launch
    huge = (1 << 64) - 16
    assert P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), huge, P.PL_F32, 0, S) == P.PL_ERR_INVALID_ARG
    assert P.purlin_all_gather(h.h, src.ptrs(), dst.ptrs(), 1 << 62, S) == P.PL_ERR_INVALID_ARG
    assert P.purlin_all_gather_v(h.h, src.ptrs(), dst.ptrs(), [1 << 63, 1 << 63, 16, 16], S) == P.PL_ERR_INVALID_ARG
    assert P.purlin_all_to_all_v(h.h, src.ptrs(), dst.ptrs(), [1 << 63] * 2 + [0] * 14, S) == P.PL_ERR_INVALID_ARG
    assert P.purlin_reduce_scatter_v(h.h, src.ptrs(), dst.ptrs(), [1 << 63, 1 << 63, 4, 4], P.PL_F32, 0,
                                     S) == P.PL_ERR_INVALID_ARG
    hh = h.h
    assert h.close() == P.PL_OK
    assert P.purlin_all_reduce(hh, src.ptrs(), dst.ptrs(), 64, P.PL_F32, 0, S) == P.PL_ERR_FINALIZED
    assert P.purlin_finalize(hh, S) == P.PL_ERR_FINALIZED
    assert src.guards_intact() and dst.guards_intact()


def test_caller_workspace_too_small_for_two_shot():
    world, n = 8, 1 << 20
    ws = torch.zeros(256 + 16, dtype=torch.uint8, device="cuda:0")   # control words + 4 flags
    h = Handle(world, ws.data_ptr(), ws.numel())
    src = RankBuffers([n * 2] * world)
    dst = RankBuffers([n * 2] * world)
    P.check(P.purlin_tune_override(h.h, {"layout": P.PL_LAYOUT_TWO_SHOT}))
    assert P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()) == P.PL_ERR_WORKSPACE
    P.check(P.purlin_tune_override(h.h, {"layout": P.PL_LAYOUT_ONE_SHOT}))
    assert P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()) == P.PL_OK
    sync()
    assert h.close() == P.PL_OK


def test_caller_workspace_two_shot():
    world, n = 8, 1 << 20
    nbytes = P.purlin_workspace_bytes(world, n * 2)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda:0")
    ins = [draw("bf16", n) for _ in range(world)]
    src = RankBuffers([n * 2] * world)
    dst = RankBuffers([n * 2] * world)
    src.upload(ins)
    h = Handle(world, ws.data_ptr(), nbytes)
    P.check(P.purlin_tune_override(h.h, {"layout": P.PL_LAYOUT_TWO_SHOT}))
    for _ in range(3):
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
    sync()
    assert h.status() == 0 and h.close() == P.PL_OK
    want = oracle.all_reduce(ins, "bf16")
    for r in range(world):
        assert np.array_equal(dst.read(r, np.uint16), want[r])


def test_consume_wait_runs_out_and_recovers():
    """A notify that never happens: the consumer gives up after the time limit,
    the device status reads TIMEOUT, and the next call on the handle is correct."""
    world, n = 4, 1 << 16
    ins = [draw("f32", n) for _ in range(world)]
    src = RankBuffers([n * 4] * world)
    dst = RankBuffers([n * 4] * world)
    src.upload(ins)
    h = Handle(world)
    P.check(P.purlin_tune_override(h.h, {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 4096}))
    P.check(P.purlin_set_wait_timeout_ns(h.h, 20_000_000))
    P.check(P.purlin_debug_drop_notify(h.h, 0))          # item 0 is a reduce that notifies
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
    sync()
    assert h.status() == P.PL_ERR_TIMEOUT
    assert h.status() == 0                                # reading clears it
    dst.fill(0)
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
    sync()
    assert h.status() == 0
    assert h.close() == P.PL_OK
    want = oracle.all_reduce(ins, "f32")
    for r in range(world):
        assert np.array_equal(bits(dst.read(r, np.float32)), bits(want[r]))


# ------------------------------------------------------ TMA bulk pipeline

BULK = {"path": P.PATH_BULK}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("world", [2, 3, 8, 11])
@pytest.mark.parametrize("stages,chunk", [(2, 4096), (3, 16384), (4, 65536)])
def test_bulk_all_reduce(dtype, world, stages, chunk):
    tune = dict(BULK, stages=stages, chunk_bytes=chunk)
    for n in (8, 1000, 65536 + 24, (1 << 20) + 8):
        for layout in (P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT):
            ins, outs = run_all_reduce(world, dtype, n, layout, tune=tune)
            want = oracle.all_reduce(ins, dtype)
            for r in range(world):
                assert np.array_equal(bits(outs[r]), bits(want[r])), (n, layout, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bulk_unaligned_and_in_place(dtype):
    E = ESZ[dtype]
    tune = dict(BULK, stages=3, chunk_bytes=8192)
    ins, outs = run_all_reduce(4, dtype, 50001, P.PL_LAYOUT_ONE_SHOT, misalign=[E, 0, 2 * E, 0], tune=tune)
    want = oracle.all_reduce(ins, dtype)
    for r in range(4):
        assert np.array_equal(bits(outs[r]), bits(want[r]))
    world, n = 8, 300000
    ins = [draw(dtype, n) for _ in range(world)]
    buf = RankBuffers([n * E] * world)
    buf.upload(ins)
    h = Handle(world)
    P.check(P.purlin_tune_override(h.h, tune))
    P.check(P.purlin_all_reduce(h.h, buf.ptrs(), buf.ptrs(), n * E, DT[dtype], 0, stream()))
    sync()
    assert h.close() == P.PL_OK
    want = oracle.all_reduce(ins, dtype)
    for r in range(world):
        assert np.array_equal(bits(buf.read(r, NP[dtype])), bits(want[r]))


@pytest.mark.parametrize("stages,chunk", [(2, 4096), (4, 32768)])
def test_bulk_copies_and_reduce_scatter(stages, chunk):
    tune = dict(BULK, stages=stages, chunk_bytes=chunk)
    world = 8
    for S in (16, 4096, 65536 + 48, (1 << 20) + 16 * 8):
        ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        outs = run_copy("ag", world, ins, S, [world * S] * world, tune=tune)
        want = oracle.all_gather(ins)
        for r in range(world):
            assert np.array_equal(outs[r], want[r])
        outs = run_copy("a2a", world, ins, S, [S] * world, tune=tune)
        want = oracle.all_to_all(ins)
        for r in range(world):
            assert np.array_equal(outs[r], want[r])
    # unaligned byte buffers fall back to the register path inside the bulk kernel
    ins = [RNG.integers(0, 256, size=1003, dtype=np.uint8) for _ in range(4)]
    outs = run_copy("ag", 4, ins, 1003, [4 * 1003] * 4, [1, 2, 3, 4], [5, 0, 7, 0], tune=tune)
    want = oracle.all_gather(ins)
    for r in range(4):
        assert np.array_equal(outs[r], want[r])
    C, c = inputs.w5_counts(world, max_count=20000, seed=4)
    a2av_in, agv_in = inputs.w5_payloads(C, c, seed=4)
    outs = run_copy("agv", world, agv_in, [int(v) * 2 for v in c], [int(c.sum()) * 2] * world, tune=tune)
    want = oracle.all_gather_v(agv_in, [int(v) for v in c])
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])
    outs = run_copy("a2av", world, a2av_in, [int(v) * 2 for v in C.reshape(-1)],
                    [int(C[:, d].sum()) * 2 for d in range(world)], tune=tune)
    want = oracle.all_to_all_v(a2av_in, C)
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])
    for dtype in ("f32", "bf16"):
        E = ESZ[dtype]
        chunk_e = 70001
        n = chunk_e * world
        ins = [draw(dtype, n) for _ in range(world)]
        src = RankBuffers([n * E] * world)
        dst = RankBuffers([chunk_e * E] * world)
        src.upload(ins)
        h = Handle(world)
        P.check(P.purlin_tune_override(h.h, tune))
        P.check(P.purlin_reduce_scatter(h.h, src.ptrs(), dst.ptrs(), n * E, DT[dtype], 0, stream()))
        sync()
        assert h.close() == P.PL_OK
        want = oracle.reduce_scatter(ins, dtype)
        for r in range(world):
            assert np.array_equal(bits(dst.read(r, NP[dtype])), bits(want[r]))
        assert dst.guards_intact()


def test_bulk_consume_wait_runs_out_and_recovers():
    world, n = 4, 1 << 16
    ins = [draw("f32", n) for _ in range(world)]
    src = RankBuffers([n * 4] * world)
    dst = RankBuffers([n * 4] * world)
    src.upload(ins)
    h = Handle(world)
    P.check(P.purlin_tune_override(h.h, dict(BULK, layout=P.PL_LAYOUT_TWO_SHOT, chunk_bytes=4096, stages=2)))
    P.check(P.purlin_set_wait_timeout_ns(h.h, 20_000_000))
    P.check(P.purlin_debug_drop_notify(h.h, 1))
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
    sync()
    assert h.status() == P.PL_ERR_TIMEOUT
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
    sync()
    assert h.status() == 0
    assert h.close() == P.PL_OK
    want = oracle.all_reduce(ins, "f32")
    for r in range(world):
        assert np.array_equal(bits(dst.read(r, np.float32)), bits(want[r]))


def test_v_variants_accept_null_for_empty_ranks():
    world = 3
    c = [5, 0, 7]
    ins = [RNG.integers(0, 256, size=v, dtype=np.uint8) for v in c]
    src = RankBuffers([max(v, 1) for v in c])
    src.upload([x if x.size else np.zeros(1, np.uint8) for x in ins])
    dst = RankBuffers([sum(c)] * world)
    sp = src.ptrs()
    sp[1] = 0                                   # a zero-byte rank may pass NULL
    h = Handle(world)
    P.check(P.purlin_all_gather_v(h.h, sp, dst.ptrs(), c, stream()))
    sync()
    want = oracle.all_gather_v(ins, c)
    for r in range(world):
        assert np.array_equal(dst.read(r), want[r])
    C = np.array([[2, 0, 1], [0, 0, 0], [3, 0, 4]])
    ins = [RNG.integers(0, 256, size=int(C[s].sum()), dtype=np.uint8) for s in range(world)]
    src = RankBuffers([max(int(C[s].sum()), 1) for s in range(world)])
    src.upload([x if x.size else np.zeros(1, np.uint8) for x in ins])
    dst = RankBuffers([max(int(C[:, d].sum()), 1) for d in range(world)])
    sp, dp = src.ptrs(), dst.ptrs()
    sp[1] = 0
    dp[1] = 0
    P.check(P.purlin_all_to_all_v(h.h, sp, dp, C.reshape(-1).tolist(), stream()))
    sync()
    want = oracle.all_to_all_v(ins, C)
    for d in (0, 2):
        assert np.array_equal(dst.read(d)[:want[d].size], want[d])
    assert P.purlin_all_gather_v(h.h, [0, 0, 0], dst.ptrs(), [1, 0, 0], stream()) == P.PL_ERR_INVALID_ARG
    assert h.close() == P.PL_OK


@pytest.mark.parametrize("path", [P.PATH_REGISTER, P.PATH_BULK])
def test_interleaved_tiles(path):
    tune = {"interleave_bytes": 16384, "path": path, "stages": 3, "chunk_bytes": 8192}
    for dtype in ("f32", "bf16"):
        ins, outs = run_all_reduce(8, dtype, (1 << 20) + 24, P.PL_LAYOUT_ONE_SHOT, tune=tune)
        want = oracle.all_reduce(ins, dtype)
        for r in range(8):
            assert np.array_equal(bits(outs[r]), bits(want[r]))
    world = 8
    C, c = inputs.w5_counts(world, max_count=30000, seed=4)
    a2av_in, agv_in = inputs.w5_payloads(C, c, seed=4)
    outs = run_copy("a2av", world, a2av_in, [int(v) * 2 for v in C.reshape(-1)],
                    [int(C[:, d].sum()) * 2 for d in range(world)], tune=tune)
    want = oracle.all_to_all_v(a2av_in, C)
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])
    outs = run_copy("agv", world, agv_in, [int(v) * 2 for v in c], [int(c.sum()) * 2] * world, tune=tune)
    want = oracle.all_gather_v(agv_in, [int(v) for v in c])
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])


@pytest.mark.parametrize("smis,dmis", [([2, 6, 10, 14], [0, 0, 0, 0]), ([0, 4, 8, 12], [2, 2, 2, 2]),
                                       ([1, 3, 5, 7], [9, 9, 9, 9])])
def test_bulk_shifted_copies(smis, dmis):
    """Sources misaligned against 16-byte destinations: the shifted bulk pipeline."""
    tune = {"path": P.PATH_BULK, "stages": 3, "chunk_bytes": 4096}
    world = 4
    for S in (17, 4096 + 2, 100000 + 6, (1 << 20) + 10):
        ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
        outs = run_copy("ag", world, ins, S, [world * S] * world, smis, dmis, tune=tune)
        want = oracle.all_gather(ins)
        for r in range(world):
            assert np.array_equal(outs[r], want[r]), (S, r)


@pytest.mark.parametrize("path", [P.PATH_REGISTER, P.PATH_BULK])
def test_trace_records_every_item(path):
    world, n = 4, 1 << 18
    ins = [draw("f32", n) for _ in range(world)]
    src = RankBuffers([n * 4] * world)
    dst = RankBuffers([n * 4] * world)
    src.upload(ins)
    tune = {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 16384, "path": path, "stages": 2}
    st, items, grid, _ = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_F32, [n * 4],
                                                src.ptrs(), dst.ptrs(), 152, tune)
    assert st == P.PL_OK
    cap = len(items) + 16
    buf = torch.zeros(8 + 32 * cap, dtype=torch.uint8, device="cuda:0")
    h = Handle(world)
    P.check(P.purlin_tune_override(h.h, tune))
    P.check(P.purlin_trace_enable(h.h, buf, buf.numel()))
    P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 4, P.PL_F32, 0, stream()))
    sync()
    P.check(P.purlin_trace_enable(h.h, None, 0))
    assert h.close() == P.PL_OK
    count, recs = P.trace_records(buf.cpu().numpy().tobytes())
    assert count == len(items)
    assert sorted(r["item"] for r in recs) == list(range(len(items)))
    for r in recs:
        assert r["end_ns"] >= r["start_ns"]
        assert r["cta"] == r["item"] % grid      # two-shot plans deal items round-robin
    want = oracle.all_reduce(ins, "f32")
    for r in range(world):
        assert np.array_equal(bits(dst.read(r, np.float32)), bits(want[r]))
