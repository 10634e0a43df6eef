"""Layout engine and tiling on the CPU: plans run by the host interpreter equal the oracle.

Covers every collective, worlds 1..16, sizes with ragged tails, unaligned
V counts, buffer addresses with mixed residues modulo 16, tiny grids (many
items per CTA) and big grids (many CTAs per piece), and the three AllReduce
layouts (all three against the one ascending fold).  Also checks the plan's
bookkeeping: CTA assignment and the SNAC rule that every wait follows its
notify in global order.
"""

import numpy as np
import pytest

import oracle
from collective_datapath_reduce_gb300 import purlin as P
from layout_interp import run_items

RNG = np.random.default_rng(1234)
QUEUED = 0xFFFFFFFF


def _describe(coll, world, dtype, sizes, sres=None, dres=None, sm=152, tune=None):
    src_addr = [0x10000 * (r + 1) + (sres[r] if sres else 0) for r in range(world)]
    dst_addr = [0x90000 * (r + 1) + (dres[r] if dres else 0) for r in range(world)]
    st, items, grid, nflags = P.purlin_plan_describe(coll, world, dtype, sizes, src_addr, dst_addr, sm, tune)
    assert st == P.PL_OK, P.purlin_status_string(st)
    assert items or sum(sizes[:1] if coll in (0, 1, 2, 3) else sizes) == 0
    for it in items:   # a fixed CTA, or any CTA (taken from the shared queue)
        assert 0 <= it["cta"] < grid or it["cta"] == QUEUED
    return items, grid, nflags


def popcount(m):
    return bin(m).count("1")


def _bytes(a):
    return np.ascontiguousarray(a).view(np.uint8).copy()


def _draw(dtype, n):
    if dtype == "f32":
        return RNG.standard_normal(n).astype(np.float32)
    return oracle.f32_to_bf16_rne(RNG.standard_normal(n).astype(np.float32))


DT = {"f32": P.PL_F32, "bf16": P.PL_BF16}
ESZ = {"f32": 4, "bf16": 2}


def _res(world, aligned):
    if aligned:
        return [0] * world
    return [int(x) for x in RNG.integers(0, 16, size=world)]


TUNES = [None, {"ctas_per_sm": 1, "min_cta_bytes": 16}, {"min_cta_bytes": 1 << 20}]
SMS = [1, 7, 152]


@pytest.mark.parametrize("world", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [P.PL_LAYOUT_ONE_SHOT, P.PL_LAYOUT_TWO_SHOT, P.PL_LAYOUT_TWO_SHOT_FUSED])
def test_all_reduce_plan(world, dtype, layout):
    E = ESZ[dtype]
    for n in (1, 7, 1000, 4096 + 3):
        for sm in SMS:
            ins = [_draw(dtype, n) for _ in range(world)]
            # element-aligned residues only (reductions need element alignment)
            sres = [int(x) * E % 16 for x in RNG.integers(0, 16, size=world)]
            dres = [int(x) * E % 16 for x in RNG.integers(0, 16, size=world)]
            tune = {"layout": layout, "chunk_bytes": 1024, "ctas_per_sm": 2, "min_cta_bytes": 64}
            items, grid, nflags = _describe(P.PL_COLL_ALL_REDUCE, world, DT[dtype], [n * E], sres, dres, sm, tune)
            outs = [np.zeros(n * E, np.uint8) for _ in range(world)]
            run_items(items, [_bytes(x) for x in ins], outs, dtype)
            want = oracle.all_reduce(ins, dtype)
            for r in range(world):
                assert np.array_equal(outs[r], _bytes(want[r])), (n, sm, r)
            if layout in (P.PL_LAYOUT_TWO_SHOT, P.PL_LAYOUT_TWO_SHOT_FUSED) and world > 1:
                assert nflags > 0
                notify_at, kinds = {}, {}
                for i, it in enumerate(items):
                    if it["notify"]:
                        notify_at[it["notify"]] = i
                    if it["wait"]:
                        # every copy follows its reduce; a CTA runs its items in
                        # increasing global order (item i on CTA i % grid)
                        assert notify_at[it["wait"]] < i
                    assert it["cta"] == i % grid
                    if it["dst_mask"] & (1 << 29):
                        # fused: reduces one tile, copies one another CTA reduced
                        assert it["wait"] and it["notify"] and it["wait"] != it["notify"]
                        assert items[notify_at[it["wait"]]]["cta"] != it["cta"]
                        kinds.setdefault(it["cta"], set()).update({True, False})
                    else:
                        kinds.setdefault(it["cta"], set()).add(popcount(it["src_mask"]) > 1)
                if len(items) >= 4 * grid and len(set(dres)) == 1:
                    # every CTA reduces and copies (none runs only one kind;
                    # copies split by destination alignment shift the order)
                    assert all(k == {True, False} for k in kinds.values())


@pytest.mark.parametrize("world", [2, 3, 8])
def test_two_shot_queue_order(world):
    """Two-shot on the shared queue: items in one global order in which every
    copy follows its reduce."""
    E = 2
    for n in (1000, 4096 + 3, 300007):
        ins = [_draw("bf16", n) for _ in range(world)]
        tune = {"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": 1024, "schedule": P.PL_SCHED_QUEUE}
        items, grid, nflags = _describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [n * E], sm=7, tune=tune)
        assert all(it["cta"] == QUEUED for it in items)
        outs = [np.zeros(n * E, np.uint8) for _ in range(world)]
        run_items(items, [_bytes(x) for x in ins], outs, "bf16")
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(outs[r], _bytes(want[r])), (n, r)
        at = {}
        for i, it in enumerate(items):
            if it["notify"]:
                at[it["notify"]] = i
            if it["wait"]:
                assert at[it["wait"]] < i


SPLIT_SRC, SPLIT_DST = 1 << 30, 1 << 31


def _ring_chunk_tiles(n, world, E, tile):
    """Tiles of the ring plan: `world` chunks of n // world elements (one more
    for the first n % world), each cut into tiles of `tile` bytes."""
    sizes = [(n // world + (1 if j < n % world else 0)) * E for j in range(world)]
    return sum(-(-b // tile) for b in sizes)


@pytest.mark.parametrize("world", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ring_all_reduce_plan(world, dtype):
    """The ring layout, run item by item on the host, gives the ascending fold
    (the oracle's AllReduce) bit for bit; its chains are ordered (every wait
    after its notify, each tile's stages one after another), every reduce
    stage adds the next rank in ascending order, the overwrite of every
    running sum waits for the read of it, and the CTAs run their items in
    increasing global order."""
    E = ESZ[dtype]
    for n in (1, 7, 1000, 4096 + 3):
        for sm in SMS:
            ins = [_draw(dtype, n) for _ in range(world)]
            sres = [int(x) * E % 16 for x in RNG.integers(0, 16, size=world)]
            dres = [int(x) * E % 16 for x in RNG.integers(0, 16, size=world)]
            tune = {"layout": P.PL_LAYOUT_RING, "chunk_bytes": 1024, "ctas_per_sm": 2}
            items, grid, nflags = _describe(P.PL_COLL_ALL_REDUCE, world, DT[dtype], [n * E], sres, dres, sm, tune)
            outs = [np.zeros(n * E, np.uint8) for _ in range(world)]
            run_items(items, [_bytes(x) for x in ins], outs, dtype)
            want = oracle.all_reduce(ins, dtype)
            for r in range(world):
                assert np.array_equal(outs[r], _bytes(want[r])), (n, sm, r)
            if world == 1:
                continue
            assert nflags > 0
            notify_at, stage_of = {}, {}
            for i, it in enumerate(items):
                ins_bits, out_bits = it["src_mask"] & 0xFFFF, it["src_mask"] >> 16
                dst_bits = it["dst_mask"] & 0xFFFF
                split_src, split_dst = bool(it["dst_mask"] & SPLIT_SRC), bool(it["dst_mask"] & SPLIT_DST)
                if it["wait"]:
                    assert it["wait"] in notify_at and notify_at[it["wait"]] < i
                    k = stage_of[it["wait"]] + 1
                else:
                    k = 1          # a tile's first stage: rank 0's input plus rank 1's
                    assert ins_bits == 3 and out_bits == 0
                if k < world:      # reduce stage k adds rank k's input to the running sum
                    assert k == 1 or ins_bits == 1 << k
                    if k > 1:
                        assert out_bits == ((3 << (k - 2)) if dtype == "bf16" else (1 << (k - 1)))
                    assert split_src == (dtype == "bf16" and k > 1)
                    assert split_dst == (dtype == "bf16" and k < world - 1)
                    assert dst_bits == ((3 << (k - 1)) if split_dst else (1 << k))
                else:              # gather stage: the finished tile passed on around the ring
                    m = k - (world - 1)
                    assert ins_bits == 0 and out_bits == 1 << ((world - 2 + m) % world)
                    assert dst_bits == 1 << ((world - 1 + m) % world) and not (split_src or split_dst)
                assert it["cta"] == i % grid
                if it["notify"]:
                    notify_at[it["notify"]] = i
                    stage_of[it["notify"]] = k
            stages = 2 * world - 2
            assert len(items) == _ring_chunk_tiles(n, world, E, 1024) * stages


def test_ring_tiles_follow_the_chunk_size():
    """Ring tiles are 64 KiB unless the caller sets chunk_bytes."""
    MI = 1 << 20
    for world, S in ((8, 1 * MI), (8, 16 * MI), (8, 64 * MI), (8, 256 * MI), (16, 64 * MI), (2, 16 * MI)):
        items, _, _ = _describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [S], tune={"layout": P.PL_LAYOUT_RING})
        assert max(int(it["len"]) for it in items) == min(65536, S // world), (world, S)
    items, _, _ = _describe(P.PL_COLL_ALL_REDUCE, 8, P.PL_BF16, [64 * MI],
                            tune={"layout": P.PL_LAYOUT_RING, "chunk_bytes": 32768})
    assert max(int(it["len"]) for it in items) == 32768


def test_ring_stages_one_wave_apart():
    """A tile's consecutive stages sit about snac_lag x grid / 2 places apart in
    the items' order (one wave of CTAs by default) while other tiles' stages
    can fill the places in between, and as far apart as the tiles allow when
    they cannot."""
    MI = 1 << 20
    for S in (4 * MI, 16 * MI, 64 * MI):
        for lag in (2, 6):
            items, grid, _ = _describe(P.PL_COLL_ALL_REDUCE, 8, P.PL_BF16, [S],
                                       tune={"layout": P.PL_LAYOUT_RING, "snac_lag": lag})
            at = {it["notify"]: i for i, it in enumerate(items) if it["notify"]}
            gaps = sorted(i - at[it["wait"]] for i, it in enumerate(items) if it["wait"])
            D = lag * grid // 2
            n_tiles = sum(1 for it in items if not it["wait"])   # first stages
            med = gaps[len(gaps) // 2]
            # with fewer tiles than D places, every tile's next stage comes
            # after the same stage of all the others
            assert min(D, n_tiles) <= med <= 2 * D, (S, lag, med, D, n_tiles)


@pytest.mark.parametrize("world", [2, 4])
def test_ring_plan_edge_cases(world):
    # the ring runs on the register path only
    st, *_ = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [4096], None, None, 152,
                                    {"layout": P.PL_LAYOUT_RING, "path": P.PATH_BULK})
    assert st == P.PL_ERR_UNSUPPORTED
    # fewer elements than ranks: empty chunks get no items, the others still complete
    items, _, _ = _describe(P.PL_COLL_ALL_REDUCE, world, P.PL_F32, [4], tune={"layout": P.PL_LAYOUT_RING})
    assert len(items) == 2 * world - 2
    # the workspace the library sizes for a handle holds the ring's flags at the table's tile size
    for S in (1 << 20, 64 << 20):
        _, _, nflags = _describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [S], tune={"layout": P.PL_LAYOUT_RING})
        assert P.purlin_workspace_bytes(world, S) >= 256 + 4 * nflags


@pytest.mark.parametrize("world", [1, 2, 5, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_plans(world, dtype):
    E = ESZ[dtype]
    for chunk in (1, 5, 333):
        for sm in SMS:
            for tune in TUNES:
                n = chunk * world
                ins = [_draw(dtype, n) for _ in range(world)]
                items, _, _ = _describe(P.PL_COLL_REDUCE_SCATTER, world, DT[dtype], [n * E], sm=sm, tune=tune)
                outs = [np.zeros(chunk * E, np.uint8) for _ in range(world)]
                run_items(items, [_bytes(x) for x in ins], outs, dtype)
                want = oracle.reduce_scatter(ins, dtype)
                for r in range(world):
                    assert np.array_equal(outs[r], _bytes(want[r]))
        # ReduceScatterV with uneven counts (some zero)
        counts = [int(c) for c in RNG.integers(0, 40, size=world)]
        if world > 1:
            counts[0] = 0
        n = sum(counts)
        ins = [_draw(dtype, n) for _ in range(world)]
        items, _, _ = _describe(P.PL_COLL_REDUCE_SCATTER_V, world, DT[dtype], [c * E for c in counts], sm=3,
                                tune={"min_cta_bytes": 16})
        outs = [np.zeros(c * E, np.uint8) for c in counts]
        run_items(items, [_bytes(x) for x in ins], outs, dtype)
        want = oracle.reduce_scatter_v(ins, counts, dtype)
        for r in range(world):
            assert np.array_equal(outs[r], _bytes(want[r]))


@pytest.mark.parametrize("world", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("aligned", [True, False])
def test_copy_plans(world, aligned):
    for S in (1, 16, 1000, 4096, 65536 + 5):
        for sm in SMS:
            tune = TUNES[int(RNG.integers(0, len(TUNES)))]
            sres, dres = _res(world, aligned), _res(world, aligned)
            ins = [RNG.integers(0, 256, size=S, dtype=np.uint8) for _ in range(world)]
            # AllGather
            items, _, _ = _describe(P.PL_COLL_ALL_GATHER, world, P.PL_U8, [S], sres, dres, sm, tune)
            outs = [np.zeros(world * S, np.uint8) for _ in range(world)]
            run_items(items, ins, outs, "u8")
            want = oracle.all_gather(ins)
            for r in range(world):
                assert np.array_equal(outs[r], want[r])
            # AllToAll (per-rank size must split into world chunks)
            S2 = (S // world) * world
            if S2:
                ins2 = [x[:S2].copy() for x in ins]
                items, _, _ = _describe(P.PL_COLL_ALL_TO_ALL, world, P.PL_U8, [S2], sres, dres, sm, tune)
                outs = [np.zeros(S2, np.uint8) for _ in range(world)]
                run_items(items, ins2, outs, "u8")
                want = oracle.all_to_all(ins2)
                for r in range(world):
                    assert np.array_equal(outs[r], want[r])


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_v_plans(world):
    for trial in range(6):
        sm = SMS[trial % 3]
        tune = TUNES[trial % len(TUNES)]
        sres, dres = _res(world, trial % 2 == 0), _res(world, trial % 2 == 0)
        c = [int(v) for v in RNG.integers(0, 300, size=world)]
        c[0] = 0 if world > 1 else c[0]
        ins = [RNG.integers(0, 256, size=c[s], dtype=np.uint8) for s in range(world)]
        items, _, _ = _describe(P.PL_COLL_ALL_GATHER_V, world, P.PL_U8, c, sres, dres, sm, tune)
        outs = [np.zeros(sum(c), np.uint8) for _ in range(world)]
        run_items(items, ins, outs, "u8")
        want = oracle.all_gather_v(ins, c)
        for r in range(world):
            assert np.array_equal(outs[r], want[r])
        C = RNG.integers(0, 200, size=(world, world))
        C[0, 0] = 0
        ins = [RNG.integers(0, 256, size=int(C[s].sum()), dtype=np.uint8) for s in range(world)]
        items, _, _ = _describe(P.PL_COLL_ALL_TO_ALL_V, world, P.PL_U8, C.reshape(-1).tolist(), sres, dres, sm, tune)
        outs = [np.zeros(int(C[:, d].sum()), np.uint8) for d in range(world)]
        run_items(items, ins, outs, "u8")
        want = oracle.all_to_all_v(ins, C)
        for r in range(world):
            assert np.array_equal(outs[r], want[r])


def test_grid_scales_with_work():
    _, g_small, _ = _describe(P.PL_COLL_ALL_GATHER, 8, P.PL_U8, [1024])
    _, g_big, _ = _describe(P.PL_COLL_ALL_GATHER, 8, P.PL_U8, [256 << 20])
    assert 1 <= g_small < g_big <= 2 * 152


def test_full_size_plans_are_balanced():
    """The workload sizes: CTAs get equal byte shares (within one 16-byte granule)."""
    for coll, world, dtype, sizes in [
        (P.PL_COLL_ALL_REDUCE, 8, P.PL_BF16, [64 << 20]),
        (P.PL_COLL_REDUCE_SCATTER, 8, P.PL_F32, [256 << 20]),
        (P.PL_COLL_ALL_GATHER, 8, P.PL_U8, [256 << 20]),
        (P.PL_COLL_ALL_TO_ALL, 8, P.PL_U8, [256 << 20]),
    ]:
        items, grid, _ = _describe(coll, world, dtype, sizes)
        if items[0]["cta"] == QUEUED:
            # queue plans: near-equal parts in global order, many per CTA
            lens = np.array([it["len"] for it in items])
            assert len(items) >= 4 * grid and lens.max() <= 1.01 * lens.mean() + 512, (coll, lens.min(), lens.max())
            for it in items:
                assert it["src_off"] % 512 == 0 and it["dst_off"] % 512 == 0
            continue
        per = np.zeros(grid, np.int64)
        nitems = np.zeros(grid, np.int64)
        for it in items:
            per[it["cta"]] += it["len"]
            nitems[it["cta"]] += 1
        # each part is the exact share rounded to 512 bytes
        assert per.max() - per.min() <= 1024 * nitems.max(), (coll, per.min(), per.max())
        assert per.max() <= 1.01 * per.mean()
        for it in items:   # every CTA share starts on a 512-byte boundary of its piece
            assert it["src_off"] % 512 == 0 and it["dst_off"] % 512 == 0


@pytest.mark.parametrize("interleave", [512, 4096, 65536])
def test_interleaved_plans(interleave):
    """Tiles dealt round-robin cover every output byte once and match the oracle."""
    tune = {"interleave_bytes": interleave}
    world = 8
    for dtype in ("f32", "bf16"):
        E = ESZ[dtype]
        n = 70001
        ins = [_draw(dtype, n) for _ in range(world)]
        items, grid, nflags = _describe(P.PL_COLL_ALL_REDUCE, world, DT[dtype], [n * E], sm=7, tune=tune)
        assert nflags == 0
        # CTA c runs parts c, c + grid, ...: its items are not contiguous in the buffer
        # unless there is one part per CTA, and consecutive items of a CTA are grid parts apart
        per = {}
        for it in items:
            per.setdefault(it["cta"], []).append(it)
        for c, its in per.items():
            offs = [it["dst_off"] for it in sorted(its, key=lambda t: t["order"])]
            assert offs == sorted(offs)
        outs = [np.zeros(n * E, np.uint8) for _ in range(world)]
        run_items(items, [_bytes(x) for x in ins], outs, dtype)
        want = oracle.all_reduce(ins, dtype)
        for r in range(world):
            assert np.array_equal(outs[r], _bytes(want[r]))
    C = RNG.integers(0, 3000, size=(world, world))
    ins = [RNG.integers(0, 256, size=int(C[s].sum()), dtype=np.uint8) for s in range(world)]
    items, _, _ = _describe(P.PL_COLL_ALL_TO_ALL_V, world, P.PL_U8, C.reshape(-1).tolist(), sm=3, tune=tune)
    outs = [np.zeros(int(C[:, d].sum()), np.uint8) for d in range(world)]
    run_items(items, ins, outs, "u8")
    want = oracle.all_to_all_v(ins, C)
    for r in range(world):
        assert np.array_equal(outs[r], want[r])
    st, *_ = P.purlin_plan_describe(P.PL_COLL_ALL_GATHER, 2, P.PL_U8, [64], tune={"interleave_bytes": 100})
    assert st == P.PL_ERR_INVALID_ARG


@pytest.mark.parametrize("part", [0, 4096, 65536])
def test_queue_plans(part):
    """Queue schedule: items in global order (part after part), same coverage as
    the static plan, every item taken by whichever CTA asks (cta = 0xFFFFFFFF)."""
    tune = {"path": P.PATH_BULK, "schedule": P.PL_SCHED_QUEUE, "interleave_bytes": part}
    world = 8
    C = RNG.integers(0, 60000, size=(world, world))
    C[0, 1] = 0
    sres, dres = _res(world, False), _res(world, False)
    src_addr = [0x1000000 * (r + 1) + sres[r] for r in range(world)]
    dst_addr = [0x9000000 * (r + 1) + dres[r] for r in range(world)]
    st, items, grid, nflags = P.purlin_plan_describe(P.PL_COLL_ALL_TO_ALL_V, world, P.PL_U8, C.reshape(-1).tolist(),
                                                     src_addr, dst_addr, 152, tune)
    assert st == P.PL_OK and nflags == 0 and 1 <= grid <= 2 * 152
    assert [it["order"] for it in items] == list(range(len(items)))
    assert all(it["cta"] == 0xFFFFFFFF for it in items)
    T = part or 256 * 1024
    total = int(C.sum())
    assert len(items) >= min(grid, total // T)
    assert max(it["len"] for it in items) <= max(2 * T, total // grid + 512)
    # global order: each destination's bytes appear in ascending offset order
    last = {}
    for it in items:
        key = it["dst_mask"]
        assert it["dst_off"] >= last.get(key, 0)
        last[key] = it["dst_off"] + it["len"]
    ins = [RNG.integers(0, 256, size=int(C[s].sum()), dtype=np.uint8) for s in range(world)]
    outs = [np.zeros(int(C[:, d].sum()), np.uint8) for d in range(world)]
    run_items(items, ins, outs, "u8")
    want = oracle.all_to_all_v(ins, C)
    for r in range(world):
        assert np.array_equal(outs[r], want[r])


def test_schedule_combinations():
    """Stream: copy plans on the bulk path.  Queue: any plan on the register
    path, copy plans on the bulk path."""
    def st(coll, dtype, sizes, **tune):
        return P.purlin_plan_describe(coll, 4, dtype, sizes, tune=tune)[0]
    AG, RS, AR = P.PL_COLL_ALL_GATHER, P.PL_COLL_REDUCE_SCATTER, P.PL_COLL_ALL_REDUCE
    for sched in (P.PL_SCHED_STREAM, P.PL_SCHED_QUEUE):
        assert st(AG, P.PL_U8, [1 << 20], path=P.PATH_BULK, schedule=sched) == P.PL_OK
        assert st(RS, P.PL_F32, [1 << 20], path=P.PATH_BULK, schedule=sched) == P.PL_ERR_UNSUPPORTED
        assert st(AR, P.PL_F32, [1 << 20], path=P.PATH_BULK, schedule=sched,
                  layout=P.PL_LAYOUT_TWO_SHOT) == P.PL_ERR_UNSUPPORTED
    assert st(AG, P.PL_U8, [1 << 20], path=P.PATH_REGISTER, schedule=P.PL_SCHED_STREAM) == P.PL_ERR_UNSUPPORTED
    for coll, dtype in ((AG, P.PL_U8), (RS, P.PL_F32), (AR, P.PL_BF16)):
        assert st(coll, dtype, [1 << 20], path=P.PATH_REGISTER, schedule=P.PL_SCHED_QUEUE) == P.PL_OK
    assert st(AR, P.PL_F32, [1 << 20], path=P.PATH_REGISTER, schedule=P.PL_SCHED_QUEUE,
              layout=P.PL_LAYOUT_TWO_SHOT) == P.PL_OK
    assert st(AG, P.PL_U8, [1 << 20], schedule=5) == P.PL_ERR_INVALID_ARG


def test_queued_two_shot_plan_orders_every_wait_after_its_notify():
    """The deadlock-freedom argument of the queue: waits point to earlier items."""
    tune = {"path": P.PATH_REGISTER, "schedule": P.PL_SCHED_QUEUE, "layout": P.PL_LAYOUT_TWO_SHOT,
            "chunk_bytes": 4096}
    for world in (2, 3, 8):
        n = 50000 * world + 7
        st, items, grid, nflags = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_F32, [n * 4], None, None,
                                                         152, tune)
        assert st == P.PL_OK and nflags > 0
        notified = {}
        for i, it in enumerate(items):
            assert it["cta"] == QUEUED and it["order"] == i
            if it["wait"]:
                assert notified.get(it["wait"], len(items)) < i
            if it["notify"]:
                notified[it["notify"]] = i
        ins = [_draw("f32", n) for _ in range(world)]
        outs = [np.zeros(n * 4, np.uint8) for _ in range(world)]
        run_items(items, [_bytes(x) for x in ins], outs, "f32")
        want = oracle.all_reduce(ins, "f32")
        for r in range(world):
            assert np.array_equal(outs[r], _bytes(want[r]))


def test_guided_queue_plans():
    """Guided queue: parts shrink from 1/(2 grid) of the work to the minimum,
    items in global order, same coverage as any other plan."""
    world = 8
    C = RNG.integers(0, 200000, size=(world, world))
    tune = {"path": P.PATH_BULK, "schedule": P.PL_SCHED_QUEUE_GUIDED, "interleave_bytes": 8192}
    sres, dres = _res(world, False), _res(world, False)
    src_addr = [0x1000000 * (r + 1) + sres[r] for r in range(world)]
    dst_addr = [0x9000000 * (r + 1) + dres[r] for r in range(world)]
    st, items, grid, _ = P.purlin_plan_describe(P.PL_COLL_ALL_TO_ALL_V, world, P.PL_U8, C.reshape(-1).tolist(),
                                                src_addr, dst_addr, 152, tune)
    assert st == P.PL_OK
    assert all(it["cta"] == QUEUED for it in items)
    W = int(C.sum())
    lens = [it["len"] for it in items]
    assert lens[0] >= W // (2 * grid) - 512 or lens[0] < 8192      # the first part is large
    assert max(lens[-20:]) <= 8192 + 512                          # the last ones are the minimum
    ins = [RNG.integers(0, 256, size=int(C[s].sum()), dtype=np.uint8) for s in range(world)]
    outs = [np.zeros(int(C[:, d].sum()), np.uint8) for d in range(world)]
    run_items(items, ins, outs, "u8")
    want = oracle.all_to_all_v(ins, C)
    for r in range(world):
        assert np.array_equal(outs[r], want[r])
    # the register path takes it too (every plan), a two-shot SNAC plan included
    st, items, _, _ = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_F32, [1 << 22], None, None, 152,
                                             {"schedule": P.PL_SCHED_QUEUE_GUIDED, "interleave_bytes": 4096})
    assert st == P.PL_OK and items[0]["len"] > items[-1]["len"]


def _header_define(name):
    import os
    import re
    from collective_datapath_reduce_gb300 import _build
    with open(os.path.join(_build.INCLUDE, "purlin_gb.h")) as f:
        return int(re.search(rf"#define {name} (\d+)u?", f.read()).group(1))


def test_default_workspace_holds_the_snac_layouts_flags():
    """The workspace a handle gets without a caller's one holds the two-shot
    and ring layouts' flags at the table's tile sizes up to the sizes the
    header states (8 ranks of 9 GiB, 16 of 4 GiB), so such calls never grow
    it; purlin_workspace_bytes sizes a workspace for a larger maximum."""
    default = _header_define("PURLIN_DEFAULT_WORKSPACE_FLAGS")
    GiB = 1 << 30
    for world, S in ((8, 9 * GiB), (16, 4 * GiB), (2, 32 * GiB), (8, 64 << 20), (3, 1000)):
        for layout in (P.PL_LAYOUT_TWO_SHOT, P.PL_LAYOUT_RING):
            st, _, _, nflags = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [S], None, None, 152,
                                                      {"layout": layout}, items=False)
            assert st == P.PL_OK
            assert nflags <= default, (world, S, layout, nflags)
            assert P.purlin_workspace_bytes(world, S) >= 256 + 4 * nflags


@pytest.mark.parametrize("world", [2, 3, 8, 16])
def test_two_shot_fused_items(world):
    """The fused two-shot layout: after a first wave of reduces, items reduce
    one tile and copy another that a different CTA reduced at least a wave
    earlier; results equal the oracle's; it runs only with store_hint 3 on
    the register path's item schedule."""
    for n, sm in ((300007, 7), (65536 * world + 5, 3), (1000, 152)):
        ins = [_draw("bf16", n) for _ in range(world)]
        tune = {"layout": P.PL_LAYOUT_TWO_SHOT_FUSED, "chunk_bytes": 4096}
        items, grid, _ = _describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [n * 2], sm=sm, tune=tune)
        outs = [np.zeros(n * 2, np.uint8) for _ in range(world)]
        run_items(items, [_bytes(x) for x in ins], outs, "bf16")
        want = oracle.all_reduce(ins, "bf16")
        for r in range(world):
            assert np.array_equal(outs[r], _bytes(want[r])), (n, sm, r)
        at = {it["notify"]: i for i, it in enumerate(items) if it["notify"]}
        fused = [i for i, it in enumerate(items) if it["dst_mask"] & (1 << 29)]
        if len(items) > 3 * grid:
            assert fused, "long plans fuse"
        for i in fused:
            j = at[items[i]["wait"]]
            assert j < i and i - j > grid and items[j]["cta"] != items[i]["cta"]
    for bad in ({"store_hint": 1}, {"schedule": P.PL_SCHED_QUEUE}, {"path": P.PATH_BULK}):
        st, *_ = P.purlin_plan_describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [1 << 20], None, None, 152,
                                        dict({"layout": P.PL_LAYOUT_TWO_SHOT_FUSED}, **bad))
        assert st == P.PL_ERR_UNSUPPORTED, bad


def _noalloc_position(G, nt, p):
    """Position p of the allocation-free AllReduce's order (the closed form its
    kernel computes, csrc/noalloc.cu): (1, tile) reduce or (2, tile) copy, the
    tiles numbered tile-major over the owners."""
    w, c = divmod(p, G)
    if w == 0:
        R, reduce_pos = c, True
    else:
        R = G + (w - 1) * (G // 2) + (c // 2 if w % 2 else (c + 1) // 2)
        reduce_pos = (w + c) % 2 == 0
    if reduce_pos and R < nt:
        return 1, R
    return 2, p - min(R, nt)


@pytest.mark.parametrize("world,n", [(8, 32 << 20), (8, 3_000_000), (3, 300001), (16, 4 * 65536 + 3), (2, 40)])
def test_noalloc_order_is_the_two_shot_order(world, n):
    """The allocation-free AllReduce computes its work positions in the kernel
    instead of uploading a plan.  Restated here, its closed form gives the
    layout engine's two-shot order (64 KiB tiles, the same even grid) item
    for item.  The sizes give every owner the same number of tiles."""
    E, T = 2, 65536
    items, grid, _ = _describe(P.PL_COLL_ALL_REDUCE, world, P.PL_BF16, [n * E],
                               tune={"layout": P.PL_LAYOUT_TWO_SHOT, "chunk_bytes": T})
    q, rem = divmod(n, world)
    start = [(o * q + min(o, rem)) * E for o in range(world + 1)]
    tiles = {-(-(start[o + 1] - start[o]) // T) for o in range(world)}
    assert len(tiles) == 1
    nt = tiles.pop() * world
    assert len(items) == 2 * nt and grid % 2 == 0
    assert grid == max(2, min(2 * 152, 2 * nt) & ~1)   # the allocation-free call's grid
    for p, it in enumerate(items):
        if popcount(it["src_mask"] & 0xFFFF) > 1:
            o = (it["dst_mask"] & 0xFFFF).bit_length() - 1
            kind = 1
        else:
            o = (it["src_mask"] >> 16).bit_length() - 1
            kind = 2
        t = (it["src_off"] - start[o]) // T
        assert (kind, t * world + o) == _noalloc_position(grid, nt, p), p
        assert it["cta"] == p % grid
