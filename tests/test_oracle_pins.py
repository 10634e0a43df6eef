"""The oracle against facts it did not produce (see pins.py for the sources)."""

import numpy as np
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle)


def test_rejects_uneven_splits():
    x = [np.zeros(5, np.float32), np.zeros(5, np.float32)]
    with pytest.raises(ValueError):
        oracle.reduce_scatter(x, "f32")
    with pytest.raises(ValueError):
        oracle.all_to_all(x)
    with pytest.raises(ValueError):
        oracle.all_reduce(x, "u8")


def _bf16_chunk(start, step):
    import torch
    torch.set_num_threads(1)
    u = np.arange(start, start + step, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    keep = ~np.isnan(f)
    mine = oracle.f32_to_bf16_rne(f)[keep]
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[keep]
    if np.array_equal(mine, ref):
        return []
    bad = np.nonzero(mine != ref)[0][:5]
    return [(hex(int(u[keep][i])), hex(int(mine[i])), hex(int(ref[i]))) for i in bad]


def test_bf16_rounding_matches_torch_on_all_patterns():
    """Every non-NaN binary32 pattern, against torch's CPU float32 -> bfloat16 (a library routine)."""
    import multiprocessing as mp
    import os
    from concurrent.futures import ProcessPoolExecutor
    step = 1 << 24
    starts = list(range(0, 1 << 32, step))
    workers = max(1, min(8, os.cpu_count() or 1))
    with ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex:
        for bad in ex.map(_bf16_chunk, starts, [step] * len(starts)):
            assert not bad, bad
