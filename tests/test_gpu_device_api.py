"""Device-side collectives (include/purlin_device.cuh) fused into a user kernel.

The example kernel (collective_datapath_reduce_gb300/examples/
fused_collectives.cu, built with the public headers only) writes the ranks'
sources inside the kernel, calls the collective, then reads the destinations.
Outputs must equal the oracle bit for bit, and the post-call reads must see
every CTA's results.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_datapath_reduce_gb300 import examples as EX
import workload_inputs as inputs

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def lib():
    return EX.load()


def run(L, which, world, ins, out_bytes, coll_frac=1.0):
    dev = torch.device("cuda", 0)
    nbytes = ins[0].nbytes
    tin = [torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).copy()).to(dev) for a in ins]
    src = [torch.zeros(nbytes, dtype=torch.uint8, device=dev) for _ in range(world)]
    dst = [torch.zeros(out_bytes, dtype=torch.uint8, device=dev) for _ in range(world)]
    post = [torch.zeros(out_bytes, dtype=torch.uint8, device=dev) for _ in range(world)]
    bar = torch.zeros(2, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    g = EX.max_grid()
    f = EX.FusedArgs()
    f.ctx.world = world
    for r in range(world):
        f.ctx.src[r] = src[r].data_ptr()
        f.ctx.dst[r] = dst[r].data_ptr()
        f.inp[r] = tin[r].data_ptr()
        f.post[r] = post[r].data_ptr()
    f.ctx.barrier = bar.data_ptr()
    f.ctx.timeout_ns = 0
    f.bytes = nbytes
    f.out_bytes = out_bytes
    f.which = which
    f.coll_blocks = max(1, int(g * coll_frac))
    f.status = status.data_ptr()
    f.work = EX.WORK_BEFORE | EX.WORK_AFTER
    for _ in range(2):       # twice: the barrier words are reused across launches
        rc = EX.launch(f, g, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, rc
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    outs = [d.cpu().numpy() for d in dst]
    for r in range(world):
        assert np.array_equal(post[r].cpu().numpy(), (outs[r].astype(np.int32) + 1).astype(np.uint8))
    return outs


@pytest.mark.parametrize("coll_frac", [1.0, 0.3])
def test_fused_all_gather_and_all_to_all(lib, coll_frac):
    rng = np.random.default_rng(31)
    world, S = 8, (1 << 20) + 48
    ins = [rng.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
    outs = run(lib, 0, world, ins, world * S, coll_frac)
    want = oracle.all_gather([x ^ 0x5A for x in ins])
    for r in range(world):
        assert np.array_equal(outs[r], want[r])
    world, S = 4, 4 * 100001
    ins = [rng.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
    outs = run(lib, 1, world, ins, S, coll_frac)
    want = oracle.all_to_all([x ^ 0x5A for x in ins])
    for r in range(world):
        assert np.array_equal(outs[r], want[r])


def test_fused_streaming_store_variants(lib):
    """The evict-first store forms, and one vector per source in flight, give the same bytes."""
    rng = np.random.default_rng(33)
    world, S = 8, (1 << 19) + 48
    ins = [rng.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
    outs = run(lib, EX.AG_STREAMING, world, ins, world * S)
    want = oracle.all_gather([x ^ 0x5A for x in ins])
    for r in range(world):
        assert np.array_equal(outs[r], want[r])
    for world in (8, 5):
        n = 200003
        ins = [inputs.to_bf16_bits(rng.standard_normal(n).astype(np.float32)) for _ in range(world)]
        want = oracle.all_reduce(ins, "bf16")
        for which in (EX.AR_BF16_STREAMING, EX.AR_BF16_U1):
            outs = run(lib, which, world, ins, n * 2)
            for r in range(world):
                assert np.array_equal(outs[r].view(np.uint16), want[r])


def test_fused_reductions(lib):
    rng = np.random.default_rng(32)
    world, n = 5, 300001
    ins = [inputs.to_bf16_bits(rng.standard_normal(n).astype(np.float32)) for _ in range(world)]
    outs = run(lib, 2, world, ins, n * 2)
    want = oracle.all_reduce(ins, "bf16")
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint16), want[r])
    world, c = 8, 70001
    ins = [rng.standard_normal(world * c).astype(np.float32) for _ in range(world)]
    outs = run(lib, 3, world, ins, c * 4)
    want = oracle.reduce_scatter(ins, "f32")
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint32), want[r].view(np.uint32))
    ins = [rng.standard_normal(100003).astype(np.float32) for _ in range(world)]
    outs = run(lib, 4, world, ins, 100003 * 4, 0.5)
    want = oracle.all_reduce(ins, "f32")
    for r in range(world):
        assert np.array_equal(outs[r].view(np.uint32), want[r].view(np.uint32))
