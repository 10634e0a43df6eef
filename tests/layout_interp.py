"""Run a plan's work items on host numpy buffers (test helper, CPU only).

This checks the layout engine and the tiling without a GPU: the items are
applied in their global order (every wait refers to an earlier notify), a
reduce item folds its sources in ascending mask-bit order in binary32 and
rounds to the output type, a copy item moves bytes.  The ring layout's bf16
items may carry a binary32 running sum as two 16-bit halves in two outputs
(destination-mask bit 30: two of the sources are those halves, low half in
the lower rank; bit 31: the two destinations receive the new sum's halves).
The result must equal the oracle's.  It is a test of which bytes go where,
not a second datapath.
"""

import numpy as np

import oracle

SPLIT_SRC, SPLIT_DST, FUSED = 1 << 30, 1 << 31, 1 << 29


QUEUED = 0xFFFFFFFF


def schedule(items):
    """The items in an order a grid of CTAs could run them: each CTA's items
    in its own order ("order" field), an item that waits only after the item
    that notifies its flag.  CTAs are stepped round-robin, each running
    whatever it can; a pass with no progress means the plan deadlocks.
    Queued items (any CTA) run in their global order."""
    if not items or "cta" not in items[0] or all(it["cta"] == QUEUED for it in items):
        return list(items)
    by_cta = {}
    for i, it in enumerate(items):
        by_cta.setdefault(it["cta"], []).append((it["order"], i))
    seqs = {c: [i for _, i in sorted(v)] for c, v in by_cta.items()}
    head = {c: 0 for c in seqs}
    flags, out = set(), []
    while len(out) < len(items):
        progress = False
        for c, seq in seqs.items():
            while head[c] < len(seq):
                it = items[seq[head[c]]]
                if it["wait"] and it["wait"] not in flags:
                    break
                out.append(it)
                if it["notify"]:
                    flags.add(it["notify"])
                head[c] += 1
                progress = True
        assert progress, "the plan's waits deadlock"
    return out


def run_items(items, ins, outs, dtype, as_given=False):
    """ins / outs: lists of uint8 arrays (rank buffers as bytes).  Items are
    applied in an order the CTAs could run them (schedule()), or as given
    (as_given: the caller orders them)."""
    world = len(outs)
    for it in (items if as_given else schedule(items)):
        n = int(it["len"])
        so, do = int(it["src_off"]), int(it["dst_off"])
        if it["dst_mask"] & FUSED:
            # two-shot fused item: reduce the tile at src_off into the
            # destination bit's output, copy the tile at dst_off from the
            # output source bit to every other output
            ranks = [r for r in range(16) if (it["src_mask"] >> r) & 1]
            ob = [r for r in range(16) if (it["src_mask"] >> (16 + r)) & 1][0]
            oa = [r for r in range(16) if (it["dst_mask"] >> r) & 1][0]
            tile = outs[ob][do:do + n].copy()
            if dtype == "f32":
                acc = oracle.fold_sum([ins[r][so:so + n].view(np.float32) for r in ranks])
                outs[oa][so:so + n] = acc.view(np.uint8)
            else:
                acc = oracle.fold_sum([oracle.bf16_bits_to_f32(ins[r][so:so + n].view(np.uint16)) for r in ranks])
                outs[oa][so:so + n] = oracle.f32_to_bf16_rne(acc).view(np.uint8)
            for d in range(world):
                if d != ob:
                    outs[d][do:do + n] = tile
            continue
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
        split_src, split_dst = bool(it["dst_mask"] & SPLIT_SRC), bool(it["dst_mask"] & SPLIT_DST)
        if len(srcs) == 1:
            val = srcs[0].copy()
        else:
            if dtype == "f32":
                cols = [s.view(np.float32) for s in srcs]
                acc = oracle.fold_sum(cols)
            else:
                if split_src:          # input sources, then the low and high halves
                    lo, hi = (s.view(np.uint16).astype(np.uint32) for s in srcs[-2:])
                    cols = [((hi << np.uint32(16)) | lo).view(np.float32)]
                    cols += [oracle.bf16_bits_to_f32(s.view(np.uint16)) for s in srcs[:-2]]
                else:
                    cols = [oracle.bf16_bits_to_f32(s.view(np.uint16)) for s in srcs]
                acc = oracle.fold_sum(cols)
            if split_dst:
                b = acc.view(np.uint32)
                outs[dsts[0]][do:do + n] = (b & np.uint32(0xFFFF)).astype(np.uint16).view(np.uint8)
                outs[dsts[1]][do:do + n] = (b >> np.uint32(16)).astype(np.uint16).view(np.uint8)
                continue
            val = acc.view(np.uint8) if dtype == "f32" else oracle.f32_to_bf16_rne(acc).view(np.uint8)
        for d in dsts:
            outs[d][do:do + n] = val
