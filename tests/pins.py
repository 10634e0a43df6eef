"""Checks that pin the CPU oracle to facts outside itself.

Every check takes the oracle module as an argument and returns normally when
the pin holds, raising AssertionError otherwise.  The oracle's own tests run
them against the real oracle; the mutation tests run them against copies of
the oracle with a plausible mistake planted (on the CPU), to show that each
mistake is caught by at least one pin.

Sources of the pins:
  * the worked all-reduce example printed by AWS Neuron NKI, "Collective
    Communication Kernels API Reference" (golden fixture);
  * the definitions there of all-gather / reduce-scatter / all-to-all along
    dim 0, applied by hand to small inputs;
  * integer-valued data, whose floating-point sums are exact whatever the order;
  * inputs whose binary32 sum depends on the order of the additions, which
    single out the ascending-rank left fold (Purlin README, "Reduction
    determinism": one fixed, repeatable result);
  * the textbook error bound of recursive summation against an exact sum;
  * algebraic invariants (AllReduce = AllGather of ReduceScatter, AllToAll is
    its own inverse, AllToAllV with transposed counts inverts AllToAllV);
  * an independently written pure-Python per-element implementation (brute.py).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _as_bits(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def eq_bits(a, b) -> bool:
    a, b = np.asarray(a), np.asarray(b)
    return a.shape == b.shape and a.dtype == b.dtype and np.array_equal(_as_bits(a), _as_bits(b))


def to_dtype(vals, dtype: str) -> np.ndarray:
    """Small exact values as rank buffers of the given dtype."""
    x = np.asarray(vals, dtype=np.float32).reshape(-1)
    if dtype == "f32":
        return x
    # exact for the small integers used by the pins: bf16 keeps 8 significant bits
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "pin value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def from_dtype(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32)
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- page values

def pin_worked_example(oracle):
    with open(os.path.join(GOLDEN, "nki_allreduce_worked_example.json")) as f:
        g = json.load(f)
    for dtype in ("f32", "bf16"):
        ins = [to_dtype(x, dtype) for x in g["inputs"]]
        outs = oracle.all_reduce(ins, dtype)
        assert len(outs) == g["world"]
        for r in range(g["world"]):
            got = from_dtype(outs[r], dtype).reshape(g["shape"])
            assert np.array_equal(got, np.asarray(g["outputs"][r], dtype=np.float32)), (dtype, r, got)


def pin_dim0_definitions(oracle):
    """The pages' dim-0 definitions applied by hand to two (2, 3) rank tensors."""
    a = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.float32)
    b = np.array([[7, 8, 9], [10, 11, 12]], dtype=np.float32)
    ins = [a.reshape(-1), b.reshape(-1)]
    # reduce-scatter: sum, then dim 0 split into 2 chunks -> rank r keeps row r of the sum
    rs = oracle.reduce_scatter(ins, "f32")
    assert np.array_equal(rs[0], [8, 10, 12]) and np.array_equal(rs[1], [14, 16, 18])
    # all-gather along dim 0: (4, 3) = rows of rank 0 then rows of rank 1, on both ranks
    ag = oracle.all_gather(ins)
    for r in range(2):
        assert np.array_equal(ag[r].reshape(4, 3), np.vstack([a, b]))
    # all-to-all along dim 0: rank i receives row i of every rank, placed in source-rank order
    aa = oracle.all_to_all(ins)
    assert np.array_equal(aa[0].reshape(2, 3), [[1, 2, 3], [7, 8, 9]])
    assert np.array_equal(aa[1].reshape(2, 3), [[4, 5, 6], [10, 11, 12]])
    # all-reduce of the same pair: element-wise sum on both ranks
    ar = oracle.all_reduce(ins, "f32")
    for r in range(2):
        assert np.array_equal(ar[r].reshape(2, 3), a + b)


# ------------------------------------------------------------ arithmetic pins

def pin_integer_exact(oracle, world=2, n=1024, seed=0):
    """Integer data: every order of additions gives the exact sum."""
    import workload_inputs as inputs
    x = inputs.w1_allreduce_ints(world, n, seed)
    exact = x.astype(np.int64).sum(axis=0)
    for dtype in ("f32", "bf16"):
        ins = [to_dtype(x[s], dtype) for s in range(world)]
        outs = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert np.array_equal(from_dtype(outs[r], dtype).astype(np.int64), exact), (dtype, r)


def pin_fold_order(oracle):
    """binary32 sums whose value depends on the order of the additions.

    1e8 is exact in binary32 and its ulp is 8, so 1e8 + 1 rounds back to 1e8.
      [1, 1e8, -1e8]      ascending: (1 + 1e8) - 1e8 = 0;  descending gives 1.
      [1e8, -1e8, 1]      ascending: 0 + 1 = 1;            descending gives 0.
      [1e8, 1, -1e8, 1]   ascending: ((1e8+1)-1e8)+1 = 1;  pairwise (1e8+1)+(-1e8+1) = 0.
    """
    cases = [([1.0, 1e8, -1e8], 0.0), ([1e8, -1e8, 1.0], 1.0), ([1e8, 1.0, -1e8, 1.0], 1.0)]
    for vals, want in cases:
        ins = [np.array([v], dtype=np.float32) for v in vals]
        got = oracle.all_reduce(ins, "f32")[0][0]
        assert got == np.float32(want), (vals, got, want)


def pin_signed_zero_and_subnormals(oracle):
    """The fold starts from rank 0's value: all -0 stays -0; subnormals are not flushed."""
    nz = np.array([-0.0], dtype=np.float32)
    out = oracle.all_reduce([nz, nz, nz], "f32")[0]
    assert out.view(np.uint32)[0] == 0x80000000
    mixed = oracle.all_reduce([nz, np.array([0.0], dtype=np.float32)], "f32")[0]
    assert mixed.view(np.uint32)[0] == 0x00000000
    tiny = np.array([1], dtype=np.uint32).view(np.float32)          # smallest subnormal
    two = oracle.all_reduce([tiny, tiny], "f32")[0]
    assert two.view(np.uint32)[0] == 2
    bnz = np.array([0x8000], dtype=np.uint16)
    assert oracle.all_reduce([bnz, bnz], "bf16")[0][0] == 0x8000
    bt = np.array([0x0001], dtype=np.uint16)                         # smallest bf16 subnormal
    assert oracle.all_reduce([bt, bt, bt], "bf16")[0][0] == 0x0003


def pin_bf16_round_cases(oracle):
    """Hand-worked rounding of binary32 patterns to bf16 (nearest, ties to even)."""
    cases = {
        0x3F800000: 0x3F80,  # 1.0 exact
        0x3F808000: 0x3F80,  # exactly half an ulp above 1.0, kept pattern even -> down
        0x3F818000: 0x3F82,  # half an ulp, kept pattern odd -> up to even
        0x3F808001: 0x3F81,  # just above half -> up
        0x3F807FFF: 0x3F80,  # just below half -> down
        0xBF808001: 0xBF81,  # negative: magnitude rounds the same way
        0x7F7FFFFF: 0x7F80,  # largest finite binary32 rounds to +inf
        0x7F7F7FFF: 0x7F7F,  # stays at the largest finite bf16
        0x00008000: 0x0000,  # tie at the smallest subnormal step, to even (zero)
        0x00018000: 0x0002,  # tie, odd kept pattern -> up
        0x7F800000: 0x7F80,  # +inf
        0xFF800000: 0xFF80,  # -inf
    }
    u = np.array(list(cases.keys()), dtype=np.uint32)
    got = oracle.f32_to_bf16_rne(u.view(np.float32))
    want = np.array(list(cases.values()), dtype=np.uint16)
    assert np.array_equal(got, want), [(hex(a), hex(b), hex(c)) for a, b, c in zip(u, got, want) if b != c]
    nan = oracle.f32_to_bf16_rne(np.array([0x7FC00000, 0xFF800001], dtype=np.uint32).view(np.float32))
    assert np.all(((nan & 0x7F80) == 0x7F80) & ((nan & 0x7F) != 0))


def pin_error_bound(oracle, world=8, n=4096, seed=11):
    """Recursive summation bound: |fold - exact| <= g_{N-1} * sum|x|, g_k = k u / (1 - k u), u = 2^-24.

    The exact sum comes from math.fsum (correctly rounded).  A dropped or
    doubled term, or a sign error, breaks the bound by orders of magnitude.
    """
    rng = np.random.default_rng(seed)
    x = (rng.random((world, n), dtype=np.float32) * 2 - 1).astype(np.float32)
    out = oracle.all_reduce([x[s] for s in range(world)], "f32")[0].astype(np.float64)
    u = 2.0 ** -24
    k = world - 1
    gamma = k * u / (1 - k * u)
    xd = x.astype(np.float64)
    for i in range(n):
        exact = math.fsum(xd[:, i])
        bound = gamma * float(np.abs(xd[:, i]).sum())
        assert abs(out[i] - exact) <= bound, (i, out[i], exact, bound)


# ---------------------------------------------------------------- invariants

def pin_invariants(oracle, seed=5):
    rng = np.random.default_rng(seed)
    for world in (1, 2, 3, 8):
        n = world * 37
        x = (rng.random((world, n), dtype=np.float32) * 2 - 1).astype(np.float32)
        for dtype in ("f32", "bf16"):
            ins = [x[s] if dtype == "f32" else oracle.f32_to_bf16_rne(x[s]) for s in range(world)]
            ar = oracle.all_reduce(ins, dtype)
            agrs = oracle.all_gather(oracle.reduce_scatter(ins, dtype))
            for r in range(world):
                assert eq_bits(ar[r], agrs[r]), (world, dtype, r)
            rsv = oracle.reduce_scatter_v(ins, [n // world] * world, dtype)
            rs = oracle.reduce_scatter(ins, dtype)
            for r in range(world):
                assert eq_bits(rsv[r], rs[r])
        b = rng.integers(0, 256, size=(world, n), dtype=np.uint8)
        bl = [b[s] for s in range(world)]
        twice = oracle.all_to_all(oracle.all_to_all(bl))
        for r in range(world):
            assert np.array_equal(twice[r], bl[r])
        # AllGatherV with equal counts is AllGather; AllToAllV with uniform counts is AllToAll
        agv = oracle.all_gather_v(bl, [n] * world)
        ag = oracle.all_gather(bl)
        a2av = oracle.all_to_all_v(bl, [[n // world] * world for _ in range(world)])
        a2a = oracle.all_to_all(bl)
        for r in range(world):
            assert np.array_equal(agv[r], ag[r]) and np.array_equal(a2av[r], a2a[r])
        # AllToAllV then AllToAllV with the transposed counts returns every buffer
        C = rng.integers(0, 6, size=(world, world))
        src = [rng.integers(0, 256, size=int(C[s].sum()), dtype=np.uint8) for s in range(world)]
        back = oracle.all_to_all_v(oracle.all_to_all_v(src, C), C.T)
        for r in range(world):
            assert np.array_equal(back[r], src[r])
        # world = 1: every collective is a copy
    one = [np.arange(6, dtype=np.float32)]
    for f in (lambda: oracle.all_reduce(one, "f32"), lambda: oracle.reduce_scatter(one, "f32"),
              lambda: oracle.all_gather(one), lambda: oracle.all_to_all(one),
              lambda: oracle.all_gather_v(one, [6]), lambda: oracle.all_to_all_v(one, [[6]])):
        assert eq_bits(f()[0], one[0])


# ------------------------------------------------------------- brute force

def pin_brute_force(oracle, seed=7):
    """Compare with the independent per-element loops on tiny inputs."""
    rng = np.random.default_rng(seed)
    for world in range(1, 6):
        for n in range(0, 18):
            x = (rng.standard_normal((world, n)) * 3).astype(np.float32)
            for dtype in ("f32", "bf16"):
                ins = [x[s] if dtype == "f32" else oracle.f32_to_bf16_rne(x[s]) for s in range(world)]
                py_ins = [[float(v) for v in b] if dtype == "f32" else [int(v) for v in b] for b in ins]
                got = oracle.all_reduce(ins, dtype)
                want = brute.all_reduce(py_ins, dtype)
                for r in range(world):
                    assert list(_as_bits(np.asarray(got[r]))) == list(_as_bits(np.asarray(want[r], dtype=got[r].dtype))), \
                        ("all_reduce", world, n, dtype)
                if n % world == 0:
                    got = oracle.reduce_scatter(ins, dtype)
                    want = brute.reduce_scatter(py_ins, dtype)
                    for r in range(world):
                        assert eq_bits(got[r], np.asarray(want[r], dtype=got[r].dtype)), ("reduce_scatter", world, n)
            b = rng.integers(0, 256, size=(world, n), dtype=np.uint8)
            bl = [b[s] for s in range(world)]
            pl = [list(map(int, b[s])) for s in range(world)]
            for r, w in enumerate(brute.all_gather(pl)):
                assert list(oracle.all_gather(bl)[r]) == w
            if n % world == 0:
                for r, w in enumerate(brute.all_to_all(pl)):
                    assert list(oracle.all_to_all(bl)[r]) == w
    # V variants: every count vector in {0..5}^N for N <= 3 (AllGatherV, ReduceScatterV),
    # and a sample of count matrices for AllToAllV
    import itertools
    for world in (1, 2, 3):
        for counts in itertools.product(range(6), repeat=world):
            bl = [rng.integers(0, 256, size=5, dtype=np.uint8) for _ in range(world)]
            pl = [list(map(int, v)) for v in bl]
            got = oracle.all_gather_v(bl, list(counts))
            for r, w in enumerate(brute.all_gather_v(pl, list(counts))):
                assert list(got[r]) == w
            n = sum(counts)
            x = (rng.standard_normal((world, n)) * 3).astype(np.float32)
            got = oracle.reduce_scatter_v([x[s] for s in range(world)], list(counts), "f32")
            want = brute.reduce_scatter_v([[float(v) for v in x[s]] for s in range(world)], list(counts), "f32")
            for r in range(world):
                assert eq_bits(got[r], np.asarray(want[r], dtype=np.float32))
        for _ in range(60 if world > 1 else 6):
            C = rng.integers(0, 6, size=(world, world))
            bl = [rng.integers(0, 256, size=int(C[s].sum()), dtype=np.uint8) for s in range(world)]
            pl = [list(map(int, v)) for v in bl]
            got = oracle.all_to_all_v(bl, C)
            for r, w in enumerate(brute.all_to_all_v(pl, C.tolist())):
                assert list(got[r]) == w


ALL_PINS = [
    pin_worked_example,
    pin_dim0_definitions,
    pin_integer_exact,
    pin_fold_order,
    pin_signed_zero_and_subnormals,
    pin_bf16_round_cases,
    pin_error_bound,
    pin_invariants,
    pin_brute_force,
]
