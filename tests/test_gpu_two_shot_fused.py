"""The fused two-shot AllReduce layout on the GPU, against the oracle.

After a first wave of reduce items, each item reduces one owner tile and, in
the same pass, copies a tile another CTA reduced a wave earlier (waiting for
its flag).  Results must equal the oracle's ascending fold bit for bit (max-ulp
0): worlds 2..16, both dtypes, ragged sizes, buffers at mixed misalignments
(whose copies go as separate items), in place, repeated calls, a dropped
notify that makes a fused item's wait run out and the next call recover, and
the 8 x 64 MiB bf16 workload.
"""

import numpy as np
import pytest
import torch

import oracle
import workload_inputs as inputs
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle, RankBuffers, bits, stream, sync
from ulp import max_ulp

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(404)
ESZ = {"f32": 4, "bf16": 2}
DT = {"f32": P.PL_F32, "bf16": P.PL_BF16}
NP = {"f32": np.float32, "bf16": np.uint16}
FUSED = {"layout": P.PL_LAYOUT_TWO_SHOT_FUSED}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


def draw(dtype, n):
    x = RNG.standard_normal(n).astype(np.float32)
    return x if dtype == "f32" else inputs.to_bf16_bits(x)


def run(world, dtype, n, tune=None, misalign=None, ins=None, h=None, in_place=False):
    E = ESZ[dtype]
    ins = ins if ins is not None else [draw(dtype, n) for _ in range(world)]
    src = RankBuffers([n * E] * world, misalign)
    dst = src if in_place else RankBuffers([n * E] * world, misalign)
    src.upload(ins)
    own = h is None
    h = h or Handle(world)
    try:
        P.check(P.purlin_tune_override(h.h, dict(FUSED, **(tune or {}))))
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * E, DT[dtype], 0, stream()), "fused")
        sync()
        assert h.status() == 0
    finally:
        if own:
            assert h.close() == P.PL_OK
    assert dst.guards_intact() and src.guards_intact()
    return ins, [dst.read(r, NP[dtype]) for r in range(world)]


@pytest.mark.parametrize("world", [2, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_matches_oracle(world, dtype):
    for n in (1, 1000, 4099, (1 << 20) + 5, (3 << 20) + 7):
        ins, outs = run(world, dtype, n, tune={"chunk_bytes": 16384})
        want = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert max_ulp(outs[r], want[r]) == 0, (n, r)
            assert np.array_equal(bits(outs[r]), bits(want[r])), (n, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_misaligned_and_in_place(dtype):
    E = ESZ[dtype]
    n, world = (1 << 20) + 3, 6
    for misalign in ([E, 2 * E, 0, 3 * E, 4 * E, 5 * E], [8] * world):
        misalign = [m % 16 - (m % 16) % E for m in misalign]
        ins, outs = run(world, dtype, n, misalign=misalign, tune={"chunk_bytes": 8192})
        want = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert np.array_equal(bits(outs[r]), bits(want[r])), (misalign, r)
    ins, outs = run(8, dtype, n, in_place=True, tune={"chunk_bytes": 8192})
    want = oracle.all_reduce(ins, dtype)
    for r in range(8):
        assert np.array_equal(bits(outs[r]), bits(want[r])), r


def test_fused_repeated_calls_and_dropped_notify():
    world, n = 8, (1 << 20) + 1
    h = Handle(world)
    try:
        for _ in range(3):
            ins, outs = run(world, "bf16", n, tune={"chunk_bytes": 8192}, h=h)
            want = oracle.all_reduce(ins, "bf16")
            for r in range(world):
                assert np.array_equal(outs[r], want[r])
        # item 0 is a reduce of the first wave: the fused item that copies its
        # tile waits, runs out, and the status reads PL_ERR_TIMEOUT
        src = RankBuffers([n * 2] * world)
        dst = RankBuffers([n * 2] * world)
        ins = [draw("bf16", n) for _ in range(world)]
        src.upload(ins)
        P.check(P.purlin_set_wait_timeout_ns(h.h, 20_000_000))
        P.check(P.purlin_debug_drop_notify(h.h, 0))
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        sync()
        assert h.status() == P.PL_ERR_TIMEOUT
        P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
        sync()
        assert h.status() == 0
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(dst.read(r, np.uint16), want[r])
    finally:
        assert h.close() == P.PL_OK


def test_fused_full_workload_8x64MiB():
    world, n = 8, 32 << 20
    x = inputs.w2_allreduce_bf16(world, n, seed=1)
    ins = [x[r] for r in range(world)]
    _, outs = run(world, "bf16", n, ins=ins)
    want = oracle.all_reduce(ins, "bf16")
    for r in range(world):
        assert max_ulp(outs[r], want[r]) == 0, r
        assert np.array_equal(outs[r], want[r]), r
    torch.cuda.empty_cache()
