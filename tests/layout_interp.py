"""Run a plan's work items on host numpy buffers (test helper, CPU only).

This checks the layout engine and the tiling without a GPU: the items are
applied in their global order (every wait refers to an earlier notify), a
reduce item folds its sources in ascending mask-bit order in binary32 and
rounds to the output type, a copy item moves bytes.  The result must equal
the oracle's.  It is a test of which bytes go where, not a second datapath.
"""

import numpy as np

import oracle


def run_items(items, ins, outs, dtype):
    """ins / outs: lists of uint8 arrays (rank buffers as bytes)."""
    for it in items:
        n = int(it["len"])
        so, do = int(it["src_off"]), int(it["dst_off"])
        srcs = []
        m = it["src_mask"]
        b = 0
        while m:
            if m & 1:
                buf = ins[b] if b < 16 else outs[b - 16]
                srcs.append(buf[so:so + n])
            m >>= 1
            b += 1
        dsts = [r for r in range(16) if (it["dst_mask"] >> r) & 1]
        if len(srcs) == 1:
            val = srcs[0].copy()
        else:
            if dtype == "f32":
                cols = [s.view(np.float32) for s in srcs]
                val = oracle.fold_sum(cols).view(np.uint8)
            else:
                cols = [oracle.bf16_bits_to_f32(s.view(np.uint16)) for s in srcs]
                val = oracle.f32_to_bf16_rne(oracle.fold_sum(cols)).view(np.uint8)
        for d in dsts:
            outs[d][do:do + n] = val
