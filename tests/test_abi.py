"""The C-ABI library loads, exports what its header declares, and rejects bad arguments (no GPU)."""

import ctypes

import pytest

from collective_datapath_reduce_gb300 import purlin as P


def test_library_exports_every_declared_symbol():
    lib = P.load()
    declared = P.declared_symbols()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), name
        assert name in P._SIGNATURES, f"binding lacks {name}"
    assert sorted(P._SIGNATURES) == declared


def test_status_strings():
    for s in range(0, 9):
        assert P.purlin_status_string(s)
    assert "time" in P.purlin_status_string(P.PL_ERR_TIMEOUT)


def test_workspace_bytes():
    assert P.purlin_workspace_bytes(0, 1 << 20) == 0
    assert P.purlin_workspace_bytes(17, 1 << 20) == 0
    small = P.purlin_workspace_bytes(8, 1 << 20)
    big = P.purlin_workspace_bytes(8, 1 << 30)
    assert 256 < small < big


def test_handle_entry_points_reject_null_handle():
    lib = P.load()
    ptrs = (ctypes.c_void_p * 2)(1, 2)
    assert lib.purlin_all_reduce(None, ptrs, ptrs, 16, P.PL_F32, 0, None) == P.PL_ERR_INVALID_ARG
    assert lib.purlin_finalize(None, None) == P.PL_ERR_INVALID_ARG
    assert lib.purlin_initialize(0, None, 0, None, None) == P.PL_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.purlin_initialize(17, None, 0, None, ctypes.byref(h)) == P.PL_ERR_INVALID_ARG


@pytest.mark.parametrize("coll,world,dtype,sizes,want", [
    (P.PL_COLL_ALL_REDUCE, 0, P.PL_F32, [16], P.PL_ERR_INVALID_ARG),
    (P.PL_COLL_ALL_REDUCE, 17, P.PL_F32, [16], P.PL_ERR_INVALID_ARG),
    (P.PL_COLL_ALL_REDUCE, 2, P.PL_U8, [16], P.PL_ERR_UNSUPPORTED),
    (P.PL_COLL_ALL_REDUCE, 2, P.PL_F32, [6], P.PL_ERR_ALIGNMENT),
    (P.PL_COLL_REDUCE_SCATTER, 3, P.PL_F32, [16], P.PL_ERR_INVALID_ARG),
    (P.PL_COLL_ALL_TO_ALL, 3, P.PL_U8, [16], P.PL_ERR_INVALID_ARG),
    (P.PL_COLL_REDUCE_SCATTER_V, 2, P.PL_BF16, [3, 4], P.PL_ERR_ALIGNMENT),
])
def test_plan_rejects(coll, world, dtype, sizes, want):
    lib = P.load()
    st = lib.purlin_plan_describe(coll, world, dtype, P._size_array(sizes), None, None, 152, None, None, 0,
                                  None, None, None)
    assert st == want


def test_plan_rejects_bad_tune():
    st, *_ = P.purlin_plan_describe(P.PL_COLL_ALL_GATHER, 2, P.PL_U8, [64], tune={"threads": 1000})
    assert st == P.PL_ERR_INVALID_ARG
    st, *_ = P.purlin_plan_describe(P.PL_COLL_ALL_GATHER, 2, P.PL_U8, [64], tune={"layout": 9})
    assert st == P.PL_ERR_UNSUPPORTED


def test_noalloc_test_hook_is_host_only_and_checks_its_tile():
    """purlin_debug_noalloc_next only records settings for the next call (no
    GPU involved); a flag index past the scratch's 16384 flags is refused."""
    assert P.purlin_debug_noalloc_next(1000, 16384) == P.PL_ERR_INVALID_ARG
    assert P.purlin_debug_noalloc_next(1000, 3) == P.PL_OK
    assert P.purlin_debug_noalloc_next(0, -1) == P.PL_OK      # cleared again
