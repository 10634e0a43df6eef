"""The seeded input generators: determinism and the tiled large-buffer generator."""

import numpy as np

import workload_inputs as inputs


def test_generators_are_seeded():
    assert np.array_equal(inputs.w2_allreduce_bf16(world=2, n=1000), inputs.w2_allreduce_bf16(world=2, n=1000))
    C1, c1 = inputs.w5_counts(8)
    C2, c2 = inputs.w5_counts(8)
    assert np.array_equal(C1, C2) and np.array_equal(c1, c2)


def test_tiled_chunks_agree_with_positions():
    for dtype, block, shift, n in (("u8", 1000, 5, 100003), ("bf16", 997, 12345, 5000), ("f32", 64, 0, 64 * 9 + 1)):
        t = inputs.Tiled(n, dtype, seed=3, shift=shift, block=block)
        starts, parts = zip(*t.chunks())
        assert list(starts) == list(range(0, n, block))
        full = np.concatenate(parts)
        assert full.size == n
        assert np.array_equal(full.view(np.uint8), t.at(np.arange(n)).view(np.uint8))
        # consecutive blocks are different rotations of the draw
        assert not np.array_equal(full[:block // 2], full[block:block + block // 2])
