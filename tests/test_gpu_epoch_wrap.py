"""The SNAC epoch counter across its wrap.

A launch of a plan with SNAC flags uses the next epoch, and a flag is ready
when it holds the launch's epoch.  Epochs run 1 .. 0xFFFFFFFF; the launch that
used 0xFFFFFFFF clears every flag of the workspace and publishes 0, so the
next launch uses 1 again and no flag value of the old cycle can look ready.
purlin_debug_set_epoch puts the counter near the end of the cycle; the
workspace is a caller tensor, so the test reads the counter and the flags
directly.  Every call's result must equal the oracle across the wrap, on the
two-shot layout (register path and bulk ring) and the ring layout.
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

RNG = np.random.default_rng(4242)
CTL_WORDS = 64          # 256 bytes of control words before the flags
EPOCH_WORD = 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


TUNES = [
    ("two_shot", {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 16384}, oracle.all_reduce),
    ("two_shot_bulk", {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 4096, "path": P.PATH_BULK, "stages": 2},
     oracle.all_reduce),
    ("ring", {"layout": P.PL_LAYOUT_RING, "chunk_bytes": 16384}, oracle.all_reduce),
    ("two_shot_fused", {"layout": P.PL_LAYOUT_TWO_SHOT_FUSED, "chunk_bytes": 4096}, oracle.all_reduce),
]


@pytest.mark.parametrize("name,tune,ref", TUNES, ids=[t[0] for t in TUNES])
def test_results_and_flags_across_the_epoch_wrap(name, tune, ref):
    world, n = 8, (1 << 18) + 5
    _, _, nflags = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [n * 2], None, None, 152, tune)[1:]
    assert nflags > 0
    ws = torch.zeros(4 * (CTL_WORDS + nflags + 1024), dtype=torch.uint8, device="cuda:0")
    words = ws.view(torch.int32)
    h = Handle(world, ws.data_ptr(), ws.numel())
    src = RankBuffers([n * 2] * world)
    dst = RankBuffers([n * 2] * world)
    try:
        P.check(P.purlin_tune_override(h.h, tune))
        # the counter never holds 0xFFFFFFFF (the next launch would take epoch 0)
        assert P.purlin_debug_set_epoch(h.h, 0xFFFFFFFF, stream()) == P.PL_ERR_INVALID_ARG
        P.check(P.purlin_debug_set_epoch(h.h, 0xFFFFFFFD, stream()))
        for k, expect in enumerate([0xFFFFFFFE, 0, 1, 2]):
            ins = [inputs.to_bf16_bits(RNG.standard_normal(n).astype(np.float32)) for _ in range(world)]
            src.upload(ins)
            dst.fill(0xEE)
            P.check(P.purlin_all_reduce(h.h, src.ptrs(), dst.ptrs(), n * 2, P.PL_BF16, 0, stream()))
            sync()
            assert h.status() == 0, k
            w = words.cpu().numpy().view(np.uint32)
            assert w[EPOCH_WORD] == expect, (k, hex(int(w[EPOCH_WORD])))
            flags = w[CTL_WORDS:]
            if expect == 0:
                assert not flags.any(), "the wrapping launch leaves every flag cleared"
            else:
                assert set(np.unique(flags[:nflags]).tolist()) <= {0, expect}, k
            want = ref(ins, "bf16")
            for r in range(world):
                assert np.array_equal(dst.read(r, np.uint16), want[r]), (k, r)
        assert dst.guards_intact() and src.guards_intact()
    finally:
        assert h.close() == P.PL_OK
