"""The torch-tensor front end: argument checks on the CPU, results on the GPU."""

import numpy as np
import pytest
import torch

import oracle
import workload_inputs as inputs
from collective_datapath_reduce_gb300 import torch_api as purlin


def test_rejects_host_tensors_without_touching_the_library():
    h = purlin.Handle(raw=None, world=2, device=torch.device("cpu"))
    xs = [torch.zeros(4), torch.zeros(4)]
    with pytest.raises(ValueError):
        purlin.all_reduce(xs, xs, h)
    with pytest.raises(ValueError):
        purlin.all_gather(xs[:1], xs[:1], h)


@pytest.fixture
def no_library(monkeypatch):
    """Any call into the C library fails the test: the checks must come first."""
    from collective_datapath_reduce_gb300 import purlin as P

    def boom(*a, **k):
        raise AssertionError("the library was called")
    for name in ("purlin_all_reduce", "purlin_reduce_scatter", "purlin_all_gather", "purlin_all_to_all",
                 "purlin_all_gather_v", "purlin_all_to_all_v", "purlin_reduce_scatter_v"):
        monkeypatch.setattr(P, name, boom)


def _bad(fn, *args, match="bytes"):
    with pytest.raises(ValueError, match=match):
        fn(*args)


def test_refuses_wrong_sized_or_typed_outputs_before_any_library_call(no_library):
    """Each output must hold exactly what the collective writes (the C ABI
    cannot see allocation sizes, so a short tensor would be overrun), in the
    inputs' dtype."""
    W = 4
    h = purlin.Handle(raw=None, world=W, device=torch.device("cpu"))
    f = lambda n, dt=torch.float32: [torch.zeros(n, dtype=dt) for _ in range(W)]
    # AllReduce: outputs of the input size, inputs all one size
    _bad(purlin.all_reduce, f(8), f(7), h)
    _bad(purlin.all_reduce, f(8)[:3] + [torch.zeros(9)], f(8), h)
    _bad(purlin.all_reduce, f(8), f(8, torch.bfloat16), h, match="dtype")
    _bad(purlin.all_reduce, f(8, torch.int32), f(8, torch.int32), h, match="float32 or bfloat16")
    # ReduceScatter: outputs of input / world elements
    _bad(purlin.reduce_scatter, f(16), f(3), h)
    _bad(purlin.reduce_scatter, f(16), f(16), h)
    _bad(purlin.reduce_scatter, f(14), f(3), h, match="equal chunks")
    _bad(purlin.reduce_scatter, f(16), f(4, torch.bfloat16), h, match="dtype")
    # AllGather: outputs of world x input
    _bad(purlin.all_gather, f(5), f(19), h)
    _bad(purlin.all_gather, f(5), f(5), h)
    # AllToAll: outputs of the input size
    _bad(purlin.all_to_all, f(8), f(4), h)
    _bad(purlin.all_to_all, f(6), f(6), h, match="equal chunks")
    # AllGatherV: every output holds the sum of the inputs
    xs = [torch.zeros(n) for n in (3, 0, 5, 1)]
    _bad(purlin.all_gather_v, xs, f(8), h)
    # AllToAllV: inputs hold their row sums, outputs their column sums
    C = [[1, 0, 2, 0], [0, 0, 0, 3], [4, 0, 0, 0], [1, 1, 1, 1]]
    rows = [torch.zeros(sum(r)) for r in C]
    cols = [torch.zeros(sum(C[s][d] for s in range(W))) for d in range(W)]
    _bad(purlin.all_to_all_v, rows, cols[:3] + [torch.zeros(1)], C, h)
    _bad(purlin.all_to_all_v, rows[:3] + [torch.zeros(9)], cols, C, h)
    _bad(purlin.all_to_all_v, rows, cols, [[1, 2]], h, match="counts")
    # ReduceScatterV: every input holds the sum of counts, output r counts[r]
    cnt = [2, 0, 3, 1]
    _bad(purlin.reduce_scatter_v, f(6), [torch.zeros(c) for c in (2, 0, 3, 2)], cnt, h)
    _bad(purlin.reduce_scatter_v, f(7), [torch.zeros(c) for c in cnt], cnt, h)
    # right sizes: the only complaint left is that host tensors are not pinned
    _bad(purlin.all_to_all_v, rows, cols, C, h, match="pinned")
    _bad(purlin.reduce_scatter_v, f(6), [torch.zeros(c) for c in cnt], cnt, h, match="pinned")
    _bad(purlin.all_gather, f(5), f(20), h, match="pinned")


@pytest.mark.gpu
def test_torch_front_end_matches_oracle():
    dev = torch.device("cuda", 0)
    world, n = 4, 100003
    rng = np.random.default_rng(5)
    h = purlin.initialize(world, dev)
    try:
        x = [inputs.to_bf16_bits(rng.standard_normal(n).astype(np.float32)) for _ in range(world)]
        xs = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev) for a in x]
        outs = [torch.empty_like(t) for t in xs]
        purlin.all_reduce(xs, outs, h, reduction_mode=purlin.ReductionMode.DETERMINISTIC)
        torch.cuda.synchronize()
        want = oracle.all_reduce(x, "bf16")
        for r in range(world):
            assert np.array_equal(outs[r].view(torch.int16).cpu().numpy().view(np.uint16), want[r])
        purlin.all_reduce(xs, xs, h)   # in place
        torch.cuda.synchronize()
        for r in range(world):
            assert np.array_equal(xs[r].view(torch.int16).cpu().numpy().view(np.uint16), want[r])
        f = [rng.standard_normal(world * 1000).astype(np.float32) for _ in range(world)]
        fs = [torch.from_numpy(a).to(dev) for a in f]
        rs = [torch.empty(1000, device=dev) for _ in range(world)]
        purlin.reduce_scatter(fs, rs, h)
        ag = [torch.empty(world * 1000, device=dev) for _ in range(world)]
        purlin.all_gather(rs, ag, h)
        aa = [torch.empty(world * 1000, device=dev) for _ in range(world)]
        purlin.all_to_all(fs, aa, h)
        torch.cuda.synchronize()
        want_rs = oracle.reduce_scatter(f, "f32")
        want_ag = oracle.all_gather(want_rs)
        want_aa = oracle.all_to_all(f)
        for r in range(world):
            assert np.array_equal(rs[r].cpu().numpy().view(np.uint32), want_rs[r].view(np.uint32))
            assert np.array_equal(ag[r].cpu().numpy().view(np.uint32), want_ag[r].view(np.uint32))
            assert np.array_equal(aa[r].cpu().numpy().view(np.uint32), want_aa[r].view(np.uint32))
        counts = [[3, 0, 5, 1], [2, 2, 2, 2], [0, 0, 0, 7], [1, 1, 0, 0]]
        send = [rng.standard_normal(sum(row)).astype(np.float32) for row in counts]
        ss = [torch.from_numpy(a).to(dev) for a in send]
        rr = [torch.empty(sum(counts[s][d] for s in range(world)), device=dev) for d in range(world)]
        purlin.all_to_all_v(ss, rr, counts, h)
        agv = [torch.empty(sum(len(a) for a in send), device=dev) for _ in range(world)]
        purlin.all_gather_v(ss, agv, h)
        torch.cuda.synchronize()
        want = oracle.all_to_all_v(send, counts)
        want_g = oracle.all_gather_v(send, [len(a) for a in send])
        for r in range(world):
            assert np.array_equal(rr[r].cpu().numpy(), want[r])
            assert np.array_equal(agv[r].cpu().numpy(), want_g[r])
    finally:
        purlin.finalize(h)


@pytest.mark.gpu
def test_torch_front_end_takes_pinned_host_tensors():
    """Pinned host tensors go to the kernels as they are (read and written in place)."""
    dev = torch.device("cuda", 0)
    world, n = 4, 50021
    rng = np.random.default_rng(6)
    h = purlin.initialize(world, dev)
    try:
        f = [rng.standard_normal(n).astype(np.float32) for _ in range(world)]
        xs = [torch.from_numpy(a.copy()).pin_memory() for a in f]
        outs = [torch.empty(n).pin_memory() for _ in range(world)]
        purlin.all_reduce(xs, outs, h)
        torch.cuda.synchronize()
        want = oracle.all_reduce(f, "f32")
        for r in range(world):
            assert np.array_equal(outs[r].numpy().view(np.uint32), want[r].view(np.uint32))
    finally:
        purlin.finalize(h)
