"""Property-based search over the layout engine's inputs (CPU only).

Random worlds, sizes, V counts, address residues, SM counts and tuning
overrides: whenever the engine accepts a call, the plan run item by item on
the host (every wait after its notify) must equal the oracle, and every item
must name a CTA of the grid or the shared queue.  Calls it refuses must be
refused with one of the documented codes.  The engine is host code shared by
every kernel, so a tiling or layout mistake shows up here without a GPU.
"""

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from collective_datapath_reduce_gb300 import purlin as P  # noqa: E402
from layout_interp import run_items  # noqa: E402

QUEUED = 0xFFFFFFFF
ESZ = {"f32": 4, "bf16": 2}
DT = {"f32": P.PL_F32, "bf16": P.PL_BF16}
ACCEPTED_REFUSALS = {P.PL_ERR_UNSUPPORTED, P.PL_ERR_INVALID_ARG, P.PL_ERR_ALIGNMENT}
SETTINGS = settings(max_examples=400, deadline=None, suppress_health_check=[HealthCheck.too_slow])


def tunes():
    return st.one_of(
        st.none(),
        st.fixed_dictionaries({}, optional={
            "ctas_per_sm": st.integers(1, 4),
            "threads": st.sampled_from([64, 128, 256, 512]),
            "unroll": st.sampled_from([1, 2, 4, 8]),
            "path": st.sampled_from([P.PATH_REGISTER, P.PATH_BULK]),
            "chunk_bytes": st.sampled_from([1024, 4096, 16384, 65536]),
            "stages": st.integers(2, 5),
            "store_hint": st.sampled_from([1, 2, 3]),
            "min_cta_bytes": st.sampled_from([16, 512, 4096, 65536]),
            "interleave_bytes": st.sampled_from([-1, 512, 4096, 16384]),
            "max_ctas": st.sampled_from([1, 7, 128]),
            "schedule": st.sampled_from([P.PL_SCHED_ITEM, P.PL_SCHED_STREAM, P.PL_SCHED_QUEUE,
                                         P.PL_SCHED_QUEUE_GUIDED]),
            "snac_lag": st.sampled_from([1, 2, 3, 5, 64]),
        }))


def _bytes(a):
    return np.ascontiguousarray(a).view(np.uint8).copy()


def _describe(coll, world, dtype, sizes, sres, dres, sm, tune):
    src = [0x10000 * (r + 1) + sres[r] for r in range(world)]
    dst = [0x900000 * (r + 1) + dres[r] for r in range(world)]
    st_, items, grid, nflags = P.purlin_plan_describe(coll, world, dtype, sizes, src, dst, sm, tune)
    if st_ != P.PL_OK:
        assert st_ in ACCEPTED_REFUSALS, P.purlin_status_string(st_)
        return None
    for it in items:
        assert it["cta"] == QUEUED or 0 <= it["cta"] < grid
        assert it["len"] > 0
    return items


@pytest.fixture(scope="module", autouse=True)
def _lib():
    P.load()


@SETTINGS
@given(world=st.integers(1, 16), n=st.integers(0, 3000), dtype=st.sampled_from(["f32", "bf16"]),
       layout=st.sampled_from([P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT, P.PL_LAYOUT_RING,
                              P.PL_LAYOUT_TWO_SHOT_FUSED]),
       sm=st.integers(1, 160), tune=tunes(), seed=st.integers(0, 2**32 - 1), data=st.data())
def test_all_reduce_plans(world, n, dtype, layout, sm, tune, seed, data):
    E = ESZ[dtype]
    rng = np.random.default_rng(seed)
    res = st.lists(st.integers(0, 15), min_size=world, max_size=world)
    sres = [r * E % 16 for r in data.draw(res)]
    dres = [r * E % 16 for r in data.draw(res)]
    t = dict(tune or {}, layout=layout)
    items = _describe(P.PL_COLL_ALL_REDUCE, world, DT[dtype], [n * E], sres, dres, sm, t)
    if items is None:
        return
    x = rng.standard_normal((world, n)).astype(np.float32)
    ins = [x[r] if dtype == "f32" else oracle.f32_to_bf16_rne(x[r]) for r in range(world)]
    outs = [np.zeros(n * E, np.uint8) for _ in range(world)]
    run_items(items, [_bytes(b) for b in ins], outs, dtype)
    want = oracle.all_reduce(ins, dtype)          # every layout gives the ascending fold
    for r in range(world):
        assert np.array_equal(outs[r], _bytes(want[r])), r


@SETTINGS
@given(world=st.integers(1, 16), chunk=st.integers(0, 700), dtype=st.sampled_from(["f32", "bf16"]),
       sm=st.integers(1, 160), tune=tunes(), seed=st.integers(0, 2**32 - 1), uneven=st.booleans(),
       data=st.data())
def test_reduce_scatter_plans(world, chunk, dtype, sm, tune, seed, uneven, data):
    E = ESZ[dtype]
    rng = np.random.default_rng(seed)
    if uneven:
        counts = data.draw(st.lists(st.integers(0, 700), min_size=world, max_size=world))
        n = sum(counts)
        coll, sizes = P.PL_COLL_REDUCE_SCATTER_V, [c * E for c in counts]
    else:
        counts = [chunk] * world
        n = chunk * world
        coll, sizes = P.PL_COLL_REDUCE_SCATTER, [n * E]
    items = _describe(coll, world, DT[dtype], sizes, [0] * world, [0] * world, sm, tune)
    if items is None:
        return
    x = rng.standard_normal((world, n)).astype(np.float32)
    ins = [x[r] if dtype == "f32" else oracle.f32_to_bf16_rne(x[r]) for r in range(world)]
    outs = [np.zeros(c * E, np.uint8) for c in counts]
    run_items(items, [_bytes(b) for b in ins], outs, dtype)
    want = oracle.reduce_scatter_v(ins, counts, dtype)
    for r in range(world):
        assert np.array_equal(outs[r], _bytes(want[r])), r


@SETTINGS
@given(world=st.integers(1, 16), S=st.integers(0, 5000), sm=st.integers(1, 160), tune=tunes(),
       kind=st.sampled_from(["ag", "a2a", "agv", "a2av"]), seed=st.integers(0, 2**32 - 1), data=st.data())
def test_copy_plans(world, S, sm, tune, kind, seed, data):
    rng = np.random.default_rng(seed)
    res = st.lists(st.integers(0, 15), min_size=world, max_size=world)
    sres, dres = data.draw(res), data.draw(res)
    if kind == "ag":
        ins = [rng.integers(0, 256, S, dtype=np.uint8) for _ in range(world)]
        items = _describe(P.PL_COLL_ALL_GATHER, world, P.PL_U8, [S], sres, dres, sm, tune)
        want = None if items is None else oracle.all_gather(ins)
        out_bytes = [world * S] * world
    elif kind == "a2a":
        S -= S % world
        ins = [rng.integers(0, 256, S, dtype=np.uint8) for _ in range(world)]
        items = _describe(P.PL_COLL_ALL_TO_ALL, world, P.PL_U8, [S], sres, dres, sm, tune)
        want = None if items is None else oracle.all_to_all(ins)
        out_bytes = [S] * world
    elif kind == "agv":
        c = data.draw(st.lists(st.integers(0, 600), min_size=world, max_size=world))
        ins = [rng.integers(0, 256, k, dtype=np.uint8) for k in c]
        items = _describe(P.PL_COLL_ALL_GATHER_V, world, P.PL_U8, c, sres, dres, sm, tune)
        want = None if items is None else oracle.all_gather_v(ins, c)
        out_bytes = [sum(c)] * world
    else:
        C = np.array(data.draw(st.lists(st.integers(0, 80), min_size=world * world, max_size=world * world)))
        C = C.reshape(world, world)
        ins = [rng.integers(0, 256, int(C[s].sum()), dtype=np.uint8) for s in range(world)]
        items = _describe(P.PL_COLL_ALL_TO_ALL_V, world, P.PL_U8, [int(v) for v in C.reshape(-1)], sres, dres, sm,
                          tune)
        want = None if items is None else oracle.all_to_all_v(ins, C)
        out_bytes = [int(C[:, d].sum()) for d in range(world)]
    if items is None:
        return
    outs = [np.zeros(b, np.uint8) for b in out_bytes]
    run_items(items, [b.copy() for b in ins], outs, "u8")
    for r in range(world):
        assert np.array_equal(outs[r], want[r]), r
