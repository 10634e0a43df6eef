"""ctypes binding of libpurlin_examples.so: a user kernel that fuses work with a
device-side collective (include/purlin_device.cuh), for tests and the benchmark."""

from __future__ import annotations

import ctypes

from . import _build

MAX_RANKS = 16
AG, A2A, AR_BF16, RS_F32, AR_F32_8, AG_STREAMING, AR_BF16_STREAMING, AR_BF16_U1 = 0, 1, 2, 3, 4, 5, 6, 7
WORK_BEFORE, WORK_AFTER = 1, 2


class Context(ctypes.Structure):
    """purlin::Context of purlin_device.cuh."""
    _fields_ = [("world", ctypes.c_int), ("src", ctypes.c_void_p * MAX_RANKS),
                ("dst", ctypes.c_void_p * MAX_RANKS), ("barrier", ctypes.c_void_p),
                ("timeout_ns", ctypes.c_ulonglong)]


class FusedArgs(ctypes.Structure):
    """Kernel arguments of examples/fused_collectives.cu."""
    _fields_ = [("ctx", Context), ("inp", ctypes.c_void_p * MAX_RANKS), ("post", ctypes.c_void_p * MAX_RANKS),
                ("bytes", ctypes.c_ulonglong), ("out_bytes", ctypes.c_ulonglong), ("which", ctypes.c_int),
                ("coll_blocks", ctypes.c_int), ("status", ctypes.c_void_p), ("work", ctypes.c_int)]


_lib = None


def load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build_examples())
        lib.purlin_example_fused_launch.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
        lib.purlin_example_fused_max_grid.argtypes = [ctypes.POINTER(ctypes.c_int)]
        if lib.purlin_example_fused_args_bytes() != ctypes.sizeof(FusedArgs):
            raise RuntimeError("FusedArgs layout does not match the example library")
        _lib = lib
    return _lib


def max_grid() -> int:
    g = ctypes.c_int()
    rc = load().purlin_example_fused_max_grid(ctypes.byref(g))
    if rc:
        raise RuntimeError(f"purlin_example_fused_max_grid failed ({rc})")
    return g.value


def launch(args: FusedArgs, grid: int, stream) -> int:
    return load().purlin_example_fused_launch(ctypes.byref(args), grid, ctypes.c_void_p(stream))
