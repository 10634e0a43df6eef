"""ctypes binding of libpurlin_gb.so: the C entry points under the same names.

Argument marshalling only: every byte of every collective is moved by the
library's CUDA kernels.  Pointers may be given as integers or as objects with
a `data_ptr()` method (torch tensors); streams as integers, `None` (legacy
default stream) or objects with a `cuda_stream` attribute.  Functions return
the C status code; out-parameters come back as extra tuple elements.  If the
library has not been built, loading it raises: there is no other code path.
"""

from __future__ import annotations

import ctypes
import os
import re

from . import _build

PL_OK = 0
PL_ERR_INVALID_ARG = 1
PL_ERR_ALIGNMENT = 2
PL_ERR_UNSUPPORTED = 3
PL_ERR_WORKSPACE = 4
PL_ERR_CUDA = 5
PL_ERR_LAUNCH = 6
PL_ERR_TIMEOUT = 7
PL_ERR_FINALIZED = 8
PL_ERR_BOUNDS = 9

PL_U8, PL_F32, PL_BF16 = 0, 1, 2
PL_DETERMINISTIC = 0

PL_COLL_ALL_REDUCE = 0
PL_COLL_REDUCE_SCATTER = 1
PL_COLL_ALL_GATHER = 2
PL_COLL_ALL_TO_ALL = 3
PL_COLL_ALL_GATHER_V = 4
PL_COLL_ALL_TO_ALL_V = 5
PL_COLL_REDUCE_SCATTER_V = 6
PL_COLL_ATOM_COPY = 7
PL_COLL_ATOM_REDUCE = 8

PL_LAYOUT_AUTO, PL_LAYOUT_ONE_SHOT, PL_LAYOUT_TWO_SHOT, PL_LAYOUT_RING, PL_LAYOUT_TWO_SHOT_FUSED = 0, 1, 2, 3, 4
PATH_REGISTER, PATH_BULK = 1, 2
PL_SCHED_ITEM, PL_SCHED_STREAM, PL_SCHED_QUEUE, PL_SCHED_QUEUE_GUIDED = 1, 2, 3, 4

MAX_WORLD = 16


class PurlinError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {purlin_status_string(status)} ({status})" if what else
                         f"{purlin_status_string(status)} ({status})")


class purlin_tune(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "layout", "ctas_per_sm", "threads", "unroll", "path", "chunk_bytes", "stages",
        "store_hint", "min_cta_bytes", "interleave_bytes", "max_ctas", "schedule", "snac_lag")]


class purlin_item(ctypes.Structure):
    _fields_ = [("src_off", ctypes.c_uint64), ("dst_off", ctypes.c_uint64), ("len", ctypes.c_uint64),
                ("src_mask", ctypes.c_uint32), ("dst_mask", ctypes.c_uint32), ("wait", ctypes.c_uint32),
                ("notify", ctypes.c_uint32), ("cta", ctypes.c_uint32), ("order", ctypes.c_uint32)]


_lib = None

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_i = ctypes.c_int
_PP = ctypes.POINTER(ctypes.c_void_p)
_SZP = ctypes.POINTER(ctypes.c_size_t)

_SIGNATURES = {
    "purlin_workspace_bytes": (_sz, [_i, _sz]),
    "purlin_initialize": (_i, [_i, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "purlin_finalize": (_i, [_vp, _vp]),
    "purlin_all_reduce": (_i, [_vp, _PP, _PP, _sz, _i, _i, _vp]),
    "purlin_reduce_scatter": (_i, [_vp, _PP, _PP, _sz, _i, _i, _vp]),
    "purlin_all_gather": (_i, [_vp, _PP, _PP, _sz, _vp]),
    "purlin_all_to_all": (_i, [_vp, _PP, _PP, _sz, _vp]),
    "purlin_all_gather_v": (_i, [_vp, _PP, _PP, _SZP, _vp]),
    "purlin_all_to_all_v": (_i, [_vp, _PP, _PP, _SZP, _vp]),
    "purlin_reduce_scatter_v": (_i, [_vp, _PP, _PP, _SZP, _i, _i, _vp]),
    "purlin_atom_copy": (_i, [_vp, _vp, _PP, _i, _sz, _vp]),
    "purlin_atom_reduce": (_i, [_vp, _PP, _i, _PP, _i, _sz, _i, _vp]),
    "purlin_status_get": (_i, [_vp, _vp, ctypes.POINTER(_i)]),
    "purlin_status_string": (ctypes.c_char_p, [_i]),
    "purlin_tune_get": (_i, [_vp, _i, _i, _sz, ctypes.POINTER(purlin_tune)]),
    "purlin_tune_override": (_i, [_vp, ctypes.POINTER(purlin_tune)]),
    "purlin_set_wait_timeout_ns": (_i, [_vp, ctypes.c_uint64]),
    "purlin_debug_limit_buffer": (_i, [_vp, _i, _i, ctypes.c_uint64]),
    "purlin_debug_set_epoch": (_i, [_vp, ctypes.c_uint32, _vp]),
    "purlin_debug_noalloc_set_epoch": (_i, [ctypes.c_uint32, _vp]),
    "purlin_debug_noalloc_next": (_i, [ctypes.c_uint64, ctypes.c_longlong]),
    "purlin_debug_drop_notify": (_i, [_vp, ctypes.c_longlong]),
    "purlin_query": (_i, [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "purlin_workspace_query": (_i, [_vp, _SZP, ctypes.POINTER(_i)]),
    "purlin_all_reduce_noalloc": (_i, [_i, _PP, _PP, _sz, _i, _vp, _vp]),
    "purlin_trace_enable": (_i, [_vp, _vp, _sz]),
    "purlin_plan_describe": (_i, [_i, _i, _i, _SZP, ctypes.POINTER(ctypes.c_uint64),
                                  ctypes.POINTER(ctypes.c_uint64), _i, ctypes.POINTER(purlin_tune),
                                  ctypes.POINTER(purlin_item), _sz, _SZP, ctypes.POINTER(_i),
                                  ctypes.POINTER(_i)]),
}


def library_path() -> str:
    return _build.LIBPATH


def load():
    """Load libpurlin_gb.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIBPATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; call __graft_entry__.build() or "
                               "python -m collective_datapath_reduce_gb300._build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def load_checking():
    """Build (if needed) and load the checking library libpurlin_gb_debug.so
    (work items checked against buffer sizes on the device).  Returns the
    library; `using(lib)` makes the wrappers of this module call it."""
    path = _build.build(debug=True)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


class using:
    """Context manager: the wrappers call `lib` (a loaded library) inside."""

    def __init__(self, lib):
        self.lib = lib

    def __enter__(self):
        global _lib
        self.prev, _lib = load(), self.lib
        return self.lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev


def declared_symbols() -> list[str]:
    """Every function the public header declares."""
    hdr = os.path.join(_build.INCLUDE, "purlin_gb.h")
    with open(hdr) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(purlin_[a-z_]+)\s*\(", text)))


# ------------------------------------------------------------- marshalling

def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return int(s.cuda_stream) or None


def _ptr_array(seq):
    vals = [_addr(x) for x in seq]
    return (ctypes.c_void_p * max(1, len(vals)))(*vals)


def _size_array(seq):
    vals = [int(x) for x in seq]
    return (ctypes.c_size_t * max(1, len(vals)))(*vals)


# ------------------------------------------------------------ entry points

def purlin_workspace_bytes(world: int, max_bytes_per_rank: int) -> int:
    return load().purlin_workspace_bytes(world, max_bytes_per_rank)


def purlin_initialize(world: int, workspace=None, workspace_bytes: int = 0, stream=None):
    h = ctypes.c_void_p()
    st = load().purlin_initialize(world, _addr(workspace) or None, workspace_bytes, _stream(stream),
                                  ctypes.byref(h))
    return st, h.value


def purlin_finalize(h, stream=None) -> int:
    return load().purlin_finalize(h, _stream(stream))


def purlin_all_reduce(h, src, dst, bytes_per_rank, dtype, mode=PL_DETERMINISTIC, stream=None) -> int:
    return load().purlin_all_reduce(h, _ptr_array(src), _ptr_array(dst), bytes_per_rank, dtype, mode,
                                    _stream(stream))


def purlin_reduce_scatter(h, src, dst, in_bytes_per_rank, dtype, mode=PL_DETERMINISTIC, stream=None) -> int:
    return load().purlin_reduce_scatter(h, _ptr_array(src), _ptr_array(dst), in_bytes_per_rank, dtype, mode,
                                        _stream(stream))


def purlin_reduce_scatter_v(h, src, dst, bytes, dtype, mode=PL_DETERMINISTIC, stream=None) -> int:
    return load().purlin_reduce_scatter_v(h, _ptr_array(src), _ptr_array(dst), _size_array(bytes), dtype,
                                          mode, _stream(stream))


def purlin_all_gather(h, src, dst, in_bytes_per_rank, stream=None) -> int:
    return load().purlin_all_gather(h, _ptr_array(src), _ptr_array(dst), in_bytes_per_rank, _stream(stream))


def purlin_all_to_all(h, src, dst, bytes_per_rank, stream=None) -> int:
    return load().purlin_all_to_all(h, _ptr_array(src), _ptr_array(dst), bytes_per_rank, _stream(stream))


def purlin_all_gather_v(h, src, dst, bytes, stream=None) -> int:
    return load().purlin_all_gather_v(h, _ptr_array(src), _ptr_array(dst), _size_array(bytes),
                                      _stream(stream))


def purlin_all_to_all_v(h, src, dst, bytes, stream=None) -> int:
    """bytes: world*world counts, row-major [src][dst]."""
    return load().purlin_all_to_all_v(h, _ptr_array(src), _ptr_array(dst), _size_array(bytes),
                                      _stream(stream))


def purlin_atom_copy(h, src, dst, nbytes, stream=None) -> int:
    return load().purlin_atom_copy(h, _addr(src), _ptr_array(dst), len(dst), nbytes, _stream(stream))


def purlin_atom_reduce(h, src, dst, nbytes, dtype, stream=None) -> int:
    return load().purlin_atom_reduce(h, _ptr_array(src), len(src), _ptr_array(dst), len(dst), nbytes, dtype,
                                     _stream(stream))


def purlin_all_reduce_noalloc(world, src, dst, bytes_per_rank, dtype, device_status=None, stream=None) -> int:
    """Allocation-free AllReduce (no handle); device_status: device int pointer or None."""
    return load().purlin_all_reduce_noalloc(world, _ptr_array(src), _ptr_array(dst), bytes_per_rank, dtype,
                                            _addr(device_status) or None, _stream(stream))


def purlin_status_get(h, stream=None):
    v = ctypes.c_int()
    st = load().purlin_status_get(h, _stream(stream), ctypes.byref(v))
    return st, v.value


def purlin_status_string(status: int) -> str:
    try:
        return load().purlin_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def purlin_tune_get(h, coll, dtype, bytes_per_rank):
    t = purlin_tune()
    st = load().purlin_tune_get(h, coll, dtype, bytes_per_rank, ctypes.byref(t))
    return st, {k: getattr(t, k) for k, _ in purlin_tune._fields_}


def make_tune(**fields) -> purlin_tune:
    t = purlin_tune()
    for k, v in fields.items():
        setattr(t, k, int(v))
    return t


def purlin_tune_override(h, tune=None) -> int:
    if tune is None:
        return load().purlin_tune_override(h, None)
    if isinstance(tune, dict):
        tune = make_tune(**tune)
    return load().purlin_tune_override(h, ctypes.byref(tune))


def purlin_set_wait_timeout_ns(h, ns: int) -> int:
    return load().purlin_set_wait_timeout_ns(h, ns)


def purlin_debug_drop_notify(h, item: int) -> int:
    return load().purlin_debug_drop_notify(h, item)


def purlin_debug_limit_buffer(h, is_output: int, rank: int, nbytes: int) -> int:
    return load().purlin_debug_limit_buffer(h, int(is_output), int(rank), int(nbytes))


def purlin_debug_set_epoch(h, epoch: int, stream=None) -> int:
    return load().purlin_debug_set_epoch(h, int(epoch), _stream(stream))


def purlin_debug_noalloc_set_epoch(epoch: int, stream=None) -> int:
    return load().purlin_debug_noalloc_set_epoch(int(epoch), _stream(stream))


def purlin_workspace_query(h):
    """(status, workspace bytes, times the library grew it)."""
    b, g = ctypes.c_size_t(), ctypes.c_int()
    st = load().purlin_workspace_query(h, ctypes.byref(b), ctypes.byref(g))
    return st, b.value, g.value


def purlin_debug_noalloc_next(timeout_ns: int = 0, drop_tile: int = -1) -> int:
    return load().purlin_debug_noalloc_next(int(timeout_ns), int(drop_tile))


def purlin_trace_enable(h, buffer=None, buffer_bytes: int = 0) -> int:
    return load().purlin_trace_enable(h, _addr(buffer) or None, buffer_bytes)


def trace_records(raw_bytes):
    """Decode a trace buffer (bytes or uint8 array): (count, list of record dicts)."""
    import numpy as np
    b = np.frombuffer(bytes(raw_bytes), dtype=np.uint8)
    count = int(b[:8].view(np.uint64)[0])
    rec = np.dtype([("start_ns", "<u8"), ("end_ns", "<u8"), ("cta", "<u4"), ("item", "<u4"),
                    ("wait_ns", "<u4"), ("len_kib", "<u4")])
    cap = (b.size - 8) // 32
    arr = b[8:8 + 32 * cap].view(rec)[:min(count, cap)]
    return count, [{k: int(r[k]) for k in rec.names} for r in arr]


def purlin_query(h):
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = load().purlin_query(h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    return st, a.value, b.value, c.value


def purlin_plan_describe(coll, world, dtype, sizes, src_addr=None, dst_addr=None, sm_count=152, tune=None,
                         items=True):
    """Returns (status, items as dicts, grid, n_flags); items=False skips the items."""
    lib = load()
    sz = _size_array(sizes)
    sa = (ctypes.c_uint64 * world)(*src_addr) if src_addr is not None else None
    da = (ctypes.c_uint64 * world)(*dst_addr) if dst_addr is not None else None
    if isinstance(tune, dict):
        tune = make_tune(**tune)
    tp = ctypes.byref(tune) if tune is not None else None
    n = ctypes.c_size_t()
    grid, nflags = ctypes.c_int(), ctypes.c_int()
    st = lib.purlin_plan_describe(coll, world, dtype, sz, sa, da, sm_count, tp, None, 0, ctypes.byref(n),
                                  ctypes.byref(grid), ctypes.byref(nflags))
    if st != PL_OK:
        return st, [], 0, 0
    if not items:
        return st, [], grid.value, nflags.value
    arr = (purlin_item * max(1, n.value))()
    st = lib.purlin_plan_describe(coll, world, dtype, sz, sa, da, sm_count, tp, arr, n.value, ctypes.byref(n),
                                  ctypes.byref(grid), ctypes.byref(nflags))
    items = [{k: getattr(arr[i], k) for k, _ in purlin_item._fields_} for i in range(n.value)]
    return st, items, grid.value, nflags.value


def check(status: int, what: str = "") -> None:
    if status != PL_OK:
        raise PurlinError(status, what)
