"""GPU test helpers: guarded rank buffers in device memory, upload and readback.

Each rank buffer is the interior of a larger torch allocation; the guard
bytes on both sides hold a fixed pattern that must survive every call (an
out-of-bounds write anywhere shows up as a changed guard).  torch only
provides memory and streams; all data movement under test is the library's.
"""

from __future__ import annotations

import numpy as np
import torch

from collective_datapath_reduce_gb300 import purlin as P

GUARD = 4096
PATTERN = 0xA5


class RankBuffers:
    """`len(sizes)` device buffers of sizes[r] bytes, each at a chosen misalignment."""

    def __init__(self, sizes, misalign=None, device="cuda:0"):
        self.sizes = [int(s) for s in sizes]
        self.misalign = [int(m) for m in (misalign or [0] * len(self.sizes))]
        self.raw = []
        for s, m in zip(self.sizes, self.misalign):
            t = torch.full((GUARD + m + s + GUARD,), PATTERN, dtype=torch.uint8, device=device)
            self.raw.append(t)

    def __len__(self):
        return len(self.sizes)

    def ptr(self, r):
        return self.raw[r].data_ptr() + GUARD + self.misalign[r]

    def ptrs(self):
        return [self.ptr(r) for r in range(len(self))]

    def view(self, r):
        o = GUARD + self.misalign[r]
        return self.raw[r][o:o + self.sizes[r]]

    def upload(self, arrays):
        for r, a in enumerate(arrays):
            b = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
            assert b.size == self.sizes[r]
            if b.size:
                self.view(r).copy_(torch.from_numpy(b.copy()))

    def fill(self, value):
        for r in range(len(self)):
            self.view(r).fill_(value)

    def read(self, r, dtype=np.uint8):
        return self.view(r).cpu().numpy().view(dtype)

    def guards_intact(self):
        for r, t in enumerate(self.raw):
            o = GUARD + self.misalign[r]
            head = t[:o]
            tail = t[o + self.sizes[r]:]
            if not bool((head == PATTERN).all()) or not bool((tail == PATTERN).all()):
                return False
        return True


class Handle:
    def __init__(self, world, workspace=None, workspace_bytes=0):
        st, self.h = P.purlin_initialize(world, workspace, workspace_bytes, stream())
        P.check(st, "purlin_initialize")
        self.world = world

    def close(self):
        if self.h is not None:
            st = P.purlin_finalize(self.h, stream())
            self.h = None
            return st
        return P.PL_OK

    def status(self):
        st, dev = P.purlin_status_get(self.h, stream())
        P.check(st, "purlin_status_get")
        return dev


def stream():
    return torch.cuda.current_stream().cuda_stream


def sync():
    torch.cuda.synchronize()


def bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a
