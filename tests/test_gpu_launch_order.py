"""Stream order around the library's launches.

Library kernels are launched with programmatic stream serialization: a call
may be scheduled while the kernel before it on the stream is finishing, and
every library kernel waits for that grid before it touches memory.  Here the
inputs of each call are produced by a torch kernel issued just before it, and
a torch kernel issued just after reads its outputs; each of many rounds
changes the values, so a call that read stale inputs, or a reader that ran
before the call finished, shows up as a mismatch.  The same chain is captured
into a CUDA graph and replayed.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_datapath_reduce_gb300 import _build
from collective_datapath_reduce_gb300 import purlin as P
from gpu_util import Handle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    P.load()


def chain(h, base, x, y, z, s, rounds, call):
    """round k: x[r] = base[r] + k (torch), call(x -> y), z[r][k] = y[r].sum() (torch)."""
    for k in range(rounds):
        for r in range(len(x)):
            torch.add(base[r], float(k), out=x[r])
        P.check(call(h, x, y, s))
        for r in range(len(y)):
            torch.sum(y[r].double(), dim=0, keepdim=True, out=z[r][k:k + 1])


@pytest.mark.parametrize("kind,n", [("all_reduce", (1 << 20) + 8), ("all_gather", (1 << 20) + 8),
                                    ("all_to_all", (1 << 20) + 8),
                                    # sizes the table runs on the streamed bulk kernel
                                    ("all_gather", (1 << 21) + 8), ("all_to_all", (1 << 22) + 8)])
def test_producer_call_consumer_chain(kind, n):
    world, rounds = 8, 12
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    base = [torch.randint(-8, 9, (n,), device=dev, generator=g).float() for _ in range(world)]
    x = [torch.empty(n, device=dev) for _ in range(world)]
    if kind == "all_reduce":
        y = [torch.empty(n, device=dev) for _ in range(world)]
        call = lambda h, a, b, s: P.purlin_all_reduce(h, a, b, n * 4, P.PL_F32, 0, s.cuda_stream)
    elif kind == "all_gather":
        y = [torch.empty(world * n, device=dev) for _ in range(world)]
        call = lambda h, a, b, s: P.purlin_all_gather(h, a, b, n * 4, s.cuda_stream)
    else:
        y = [torch.empty(n, device=dev) for _ in range(world)]
        call = lambda h, a, b, s: P.purlin_all_to_all(h, a, b, n * 4, s.cuda_stream)
    z = [torch.zeros(rounds, dtype=torch.float64, device=dev) for _ in range(world)]
    h = Handle(world)
    s = torch.cuda.Stream()
    try:
        with torch.cuda.stream(s):
            chain(h.h, base, x, y, z, s, rounds, call)
            s.synchronize()
            bh = [b.cpu().numpy() for b in base]
            for k in range(rounds):
                ins = [b + np.float32(k) for b in bh]
                want = {"all_reduce": lambda: oracle.all_reduce(ins, "f32"),
                        "all_gather": lambda: oracle.all_gather(ins),
                        "all_to_all": lambda: oracle.all_to_all([a.view(np.uint8) for a in ins])}[kind]()
                for r in range(world):
                    w = want[r] if kind != "all_to_all" else want[r].view(np.float32)
                    # integer-valued data: every sum is exact in any order
                    assert float(z[r][k]) == float(w.astype(np.float64).sum()), (kind, k, r)
            # the same chain in a CUDA graph, replayed twice
            for t in z:
                t.zero_()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                chain(h.h, base, x, y, z, s, rounds, call)
            for _ in range(2):
                graph.replay()
                s.synchronize()
                for k in range(rounds):
                    ins = [b + np.float32(k) for b in bh]
                    tot = sum(float(a.astype(np.float64).sum()) for a in ins)
                    if kind == "all_reduce":
                        expect = [tot] * world
                    elif kind == "all_gather":
                        expect = [tot] * world
                    else:
                        w = oracle.all_to_all([a.view(np.uint8) for a in ins])
                        expect = [float(a.view(np.float32).astype(np.float64).sum()) for a in w]
                    for r in range(world):
                        assert float(z[r][k]) == expect[r], ("graph", kind, k, r)
            del graph
        assert h.status() == 0
    finally:
        assert h.close() == P.PL_OK
