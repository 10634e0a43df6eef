"""SNAC schedules run on the CPU with one thread per CTA (no GPU).

The two-shot and ring AllReduce plans deal their items round-robin to the CTAs; each
item that consumes a flag waits (bounded) until the item that notifies it has
run.  Here every CTA is a Python thread that walks its items in the kernel's
order, waits on flags set by other threads, and applies the item to host
buffers.  The plan must finish and match the oracle for any grid size; with
one notify dropped the consumer must time out, record the failure, and every
thread must still return (the device kernel's behaviour, on the host).
"""

import threading

import numpy as np
import pytest

import oracle
from collective_datapath_reduce_gb300 import purlin as P
from layout_interp import run_items


def run_threads(items, grid, ins, outs, dtype, drop=None, timeout=5.0):
    flags = {}
    cond = threading.Condition()
    status = {"failed": False}
    by_cta = {}
    for i, it in enumerate(items):
        by_cta.setdefault(it["cta"], []).append((i, it))

    def cta(c):
        for i, it in by_cta.get(c, []):
            with cond:
                if status["failed"]:
                    return
                if it["wait"]:
                    ok = cond.wait_for(lambda: flags.get(it["wait"]) or status["failed"], timeout=timeout)
                    if not ok or status["failed"]:
                        status["failed"] = True
                        cond.notify_all()
                        return
            run_items([it], ins, outs, dtype, as_given=True)   # the item's data movement
            if it["notify"] and i != drop:
                with cond:
                    flags[it["notify"]] = True
                    cond.notify_all()

    threads = [threading.Thread(target=cta, args=(c,)) for c in range(grid)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=4 * timeout)
        assert not t.is_alive(), "a CTA thread did not return"
    return not status["failed"]


LAYOUTS = [(P.PL_LAYOUT_TWO_SHOT, oracle.all_reduce), (P.PL_LAYOUT_RING, oracle.all_reduce)]


@pytest.mark.parametrize("sm", [1, 3, 16])
@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("layout,ref", LAYOUTS, ids=["two_shot", "ring"])
def test_snac_schedule_completes_under_threads(sm, world, layout, ref):
    """Two-shot: one wait per copy.  Ring: a chain of 2 (world - 1) stages per
    tile, whose running sums are overwritten later in the same chain."""
    rng = np.random.default_rng(world * 100 + sm)
    n = 5000 * world + 3
    ins = [oracle.f32_to_bf16_rne(rng.standard_normal(n).astype(np.float32)) for _ in range(world)]
    tune = {"layout": layout, "chunk_bytes": 1024, "ctas_per_sm": 2}
    st, items, grid, nflags = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [n * 2], None, None,
                                                     sm, tune)
    assert st == P.PL_OK and nflags > 0
    outs = [np.zeros(n * 2, np.uint8) for _ in range(world)]
    assert run_threads(items, grid, [x.view(np.uint8).copy() for x in ins], outs, "bf16")
    want = ref(ins, "bf16")
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])


def test_dropped_notify_times_out_and_every_cta_returns():
    world, n = 4, 20000
    ins = [np.ones(n, np.float32) for _ in range(world)]
    tune = {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 4096}
    st, items, grid, _ = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_F32, [n * 4], None, None, 4, tune)
    assert st == P.PL_OK
    notifier = next(i for i, it in enumerate(items) if it["notify"])
    outs = [np.zeros(n * 4, np.uint8) for _ in range(world)]
    ok = run_threads(items, grid, [x.view(np.uint8).copy() for x in ins], outs, "f32", drop=notifier, timeout=0.5)
    assert not ok
