// Layout engine and tiling (host only).
//
// Step 1, layouts: each collective becomes a list of pieces (see plan.h).
//   AllReduce, one-shot  (Iris docs, "Device Context", all_reduce_one_shot:
//       every rank reads all ranks and reduces locally): one reduce piece over
//       the whole buffer, sources = all inputs, destinations = all outputs.
//   AllReduce, two-shot  (same page, all_reduce_two_shot: each rank reduces
//       only its share, then the result is scattered, with ready flags):
//       rank o owns the o-th of world near-equal element ranges; per tile t of
//       that range a reduce piece writes out[o] and raises flag (o, t), and a
//       copy piece waits on the flag and copies out[o] to every other output.
//   AllReduce, ring  (same page, all_reduce_ring: a running sum handed from
//       rank to rank, then the result passed around the ring): per tile,
//       2 (world - 1) stages chained by flags: world - 1 reduce pieces that
//       add ranks 1 .. world-1 in ascending order to the binary32 sum the
//       previous stage left in the outputs, then world - 1 copies that pass
//       the finished tile around the ring.
//   ReduceScatter  (NKI, reduce_scatter_hbm_kernel): piece r reduces chunk r of
//       all inputs into out[r].
//   AllGather      (NKI, all_gather_hbm_kernel): piece s copies in[s] to offset
//       s*S of every output (one read, world writes).
//   AllToAll       (NKI, all_to_all_hbm_kernel): piece (s, d) copies chunk d of
//       in[s] to chunk s of out[d].
//   V variants     (Purlin README summary): the same pieces at prefix-sum
//       displacements of the given byte counts.
// Step 2, tiling: pieces are concatenated into one byte space that is cut
// into `grid` contiguous, equal shares (Iris docs, reduce_scatter:
// contiguous work distribution), one per persistent CTA.  Plans with SNAC
// flags keep each piece whole and deal the items out round-robin instead, so
// that producers and consumers of a flag run at about the same time.
#include "plan.h"

#include <algorithm>
#include <cstring>
#include <sstream>

#include "purlin_gb.h"

namespace pl {

namespace {

struct Piece {
  uint64_t src_off, dst_off, len;
  uint32_t src_mask, dst_mask;
  uint32_t wait, notify;
};

constexpr uint64_t kMaxItemBytes = 1ull << 30;
// Queue schedule without interleave_bytes: parts of about this size.
constexpr uint64_t kQueuePartBytes = 256 * 1024;
// CTA shares are cut at multiples of 512 bytes from a piece's start, so that a
// warp's 32 x 16-byte vectors cover whole 128-byte lines and 32-byte sectors
// (a cut at 16 bytes leaves every warp straddling one extra line and two
// partial sectors, which cost DRAM fills).
constexpr uint64_t kSplitGranule = 512;

inline uint32_t all_ranks(int world) { return (world >= 32) ? 0xFFFFFFFFu : ((1u << world) - 1u); }
inline uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
inline int popcount32(uint32_t x) { return __builtin_popcount(x); }

bool is_reduce_coll(int coll) {
  return coll == kAllReduce || coll == kReduceScatter || coll == kReduceScatterV ||
         coll == kAtomReduce;
}

// Split a piece whose destinations do not all share one address residue
// modulo 16 into one piece per residue class (the Atoms store one vector to
// every destination of an item and need them co-aligned).
void push_grouped(std::vector<Piece>& out, const Piece& p, const uint8_t* dst_res) {
  if (p.len == 0) return;
  uint32_t left = p.dst_mask;
  while (left) {
    int first = __builtin_ctz(left);
    uint32_t res = (dst_res[first] + p.dst_off) & 15u;
    uint32_t group = 0;
    for (uint32_t m = left; m; m &= m - 1) {
      int r = __builtin_ctz(m);
      if (((dst_res[r] + p.dst_off) & 15u) == res) group |= 1u << r;
    }
    Piece q = p;
    q.dst_mask = group;
    out.push_back(q);
    left &= ~group;
  }
}

}  // namespace

int elem_size(int dtype) { return dtype == kF32 ? 4 : (dtype == kBF16 ? 2 : 1); }

size_t n_sizes(int coll, int world) {
  switch (coll) {
    case kAllGatherV:
    case kReduceScatterV:
      return (size_t)world;
    case kAllToAllV:
      return (size_t)world * (size_t)world;
    case kAtomReduce:
      return 3;
    default:
      return 1;
  }
}

// Tuning table, from the sweeps measured on a GB300 (152 SMs, HBM3e):
// `bytes_per_rank` is the per-rank size the collective moves (for the V
// variants, their total divided by the world).  Summary of what won:
//   AllReduce   (8 ranks) register path, 512 threads; from 8 MiB per rank 128 CTAs with
//               one contiguous share each and evict-first stores (96% of the
//               measured copy bandwidth at 8 x 64 MiB bf16, 99.9% at 8 x 256
//               MiB; one CTA per SM or more gave 90-92%: fewer concurrent DRAM
//               streams win); the fewest bytes per CTA stay at 512 so small
//               calls spread over many CTAs.  2 ranks: 3 CTAs of 256 threads
//               per SM; more than 8: 256 CTAs of 256 threads.
//   ReduceScatter  from 64 MiB per rank the TMA bulk ring (2 slots x 32 KiB
//               per source), above the copy bandwidth from 128 MiB (the
//               traffic is 8 reads per write); below, the register path with
//               3 CTAs of 256 threads per SM (10% ahead of the ring at 16-32
//               MiB), write-back stores from 4 MiB.
//   AllGather   from 8 MiB per rank the streamed bulk ring fed from the
//               shared item queue in 16 KiB parts (6904 against 6466 GB/s for
//               register copies at 8 x 256 MiB, 6361 against 5572 at 8 MiB);
//               from 4 MiB register copies on 128 CTAs of 512 threads with
//               evict-first stores (5756 against 5646 at 4 MiB).  AllGatherV
//               (misaligned pieces): the guided queue on 128 CTAs, parts of
//               32 KiB shrinking to 8 KiB (5889 against 5681 item by item for
//               equal 32 KiB parts; the guided parts 1% faster again).
//   AllToAll    from 16 MiB per rank the queue in 64 KiB parts, 5 slots (7096
//               against 6864 item by item at 256 MiB, 6800 against 6557 at 64
//               MiB); AllToAllV from 32 MiB the guided queue (parts of
//               256 KiB shrinking to 64 KiB), 4 slots.  Below, register copies:
//               write-back stores from 2 MiB (17-23% ahead of streaming
//               stores at 2-8 MiB), streaming stores below.
//   Copy Atom, one destination: from 32 MiB the queue in 64 KiB parts (6973
//               against 6762 GB/s item by item at 1 GiB); from 4 MiB, 8
//               vectors per thread, write-back stores.
Tune tune_table(int coll, int world, int dtype, uint64_t bytes_per_rank) {
  (void)dtype;
  const uint64_t S = bytes_per_rank;
  constexpr uint64_t KiB = 1024, MiB = 1024 * 1024;
  Tune t;
  t.layout = kOneShot;
  t.path = kPathRegister;
  t.threads = 256;
  t.ctas_per_sm = 2;
  t.unroll = 4;
  t.chunk_bytes = 32 * 1024;
  t.stages = 3;
  t.store_hint = 1;
  t.min_cta_bytes = 512;
  t.schedule = kSchedItem;
  t.snac_lag = 2;  // two-shot: copies at least one wave of CTAs after their reduce
  switch (coll) {
    case kAllReduce:
    case kAtomReduce:
      t.unroll = world <= 4 ? 2 : 1;
      t.chunk_bytes = 64 * 1024;  // two-shot tile
      t.threads = 512;
      if (S >= 8 * MiB && world <= 2) {
        // two sources: few bytes in flight per thread, so many more CTAs
        // (6057 against 5082 GB/s for the 128-CTA setting at 2 x 64 MiB)
        t.threads = 256;
        t.ctas_per_sm = 3;
        t.store_hint = 2;
      } else if (S >= 8 * MiB && world > 8) {
        // more than 8 sources: CTAs of 256 threads (the generic-count kernel's
        // bound), 256 of them (6612 against 5312 GB/s for 128 at 16 x 64 MiB)
        t.threads = 256;
        t.max_ctas = 256;
        t.store_hint = 2;
      } else if (S >= 8 * MiB) {
        // 128 CTAs of 512 threads, one contiguous share each, evict-first
        // stores: fewer concurrent DRAM streams than one CTA per SM
        t.max_ctas = 128;
        t.store_hint = 2;
      }
      break;
    case kReduceScatter:
    case kReduceScatterV:
      t.unroll = world <= 4 ? 2 : 1;
      if (S >= 64 * MiB) {
        // the bulk ring: level with the register path when calls run back to
        // back, and unaffected by what the L2 held before the call (after an
        // L2-sized write the register path loses 7% at 8 x 256 MiB fp32)
        t.path = kPathBulk;
        t.ctas_per_sm = 1;
        t.stages = 2;
        t.chunk_bytes = 32 * 1024;
      } else {
        // register path, three CTAs per SM, evict-first stores (against the
        // bulk ring: 6216 / 5567 GB/s at 8 x 16 MiB fp32, 6750 / 6163 at 32 MiB);
        // from 4 MiB with write-back stores (a CUDA graph of 10 calls after an
        // L2-sized write: 3-6% ahead at 4-32 MiB, fp32 and bf16; 1-2% for the
        // uneven chunks of ReduceScatterV at 36-40 MiB)
        t.ctas_per_sm = 3;
        t.store_hint = S >= 4 * MiB ? 1 : 2;
      }
      break;
    case kAllGather:
    case kAllGatherV:
    case kAtomCopy:
      if (coll == kAtomCopy && world == 1 && S >= 4 * MiB) {
        // one destination: one store per load, so more bytes in flight per
        // thread; from 32 MiB the bulk ring fed from the shared queue
        if (S >= 32 * MiB) {
          t.path = kPathBulk;
          t.ctas_per_sm = 1;
          t.stages = 4;
          t.schedule = kSchedQueue;
          t.interleave_bytes = 64 * 1024;
        } else {
          // write-back stores: 5.01 against 5.27 us at 8 MiB (graph of 10 calls)
          t.threads = 512;
          t.unroll = 8;
          t.max_ctas = 128;
          t.store_hint = 1;
        }
      } else if (S >= 4 * MiB && coll == kAllGatherV) {
        // AllGatherV pieces are mostly misaligned: shifted bulk copies from
        // the guided queue (parts of 32 KiB shrinking to 8 KiB at the end:
        // 66.0 against 66.7 us for equal 32 KiB parts), 128 CTAs
        t.path = kPathBulk;
        t.ctas_per_sm = 1;
        t.max_ctas = 128;
        t.stages = 3;
        t.chunk_bytes = 32 * 1024;
        t.schedule = kSchedQueueGuided;
        t.interleave_bytes = 8 * 1024;
      } else if (S >= 8 * MiB && coll == kAllGather) {
        // one bulk load, `world` bulk stores per chunk, one CTA per SM, parts
        // from the shared queue: 16 KiB with 3 slots for 8 ranks, 64 KiB with
        // 4 slots for up to 4 (6283 against 4644 GB/s at 2 x 64 MiB)
        t.path = kPathBulk;
        t.ctas_per_sm = 1;
        t.stages = world <= 4 ? 4 : 3;
        t.chunk_bytes = 32 * 1024;
        t.schedule = kSchedQueue;
        t.interleave_bytes = world <= 4 ? 64 * 1024 : 16 * 1024;
      } else if (S >= 4 * MiB) {
        // one load, eight stores per vector: like the AllReduce, 128 CTAs of
        // 512 threads with evict-first stores
        t.threads = 512;
        t.max_ctas = 128;
        t.store_hint = 2;
      } else if (S >= 256 * KiB) {
        t.threads = 512;
        t.min_cta_bytes = 2 * 1024;
      }
      break;
    case kAllToAll:
    case kAllToAllV:
      if (coll == kAllToAllV && S >= 32 * MiB) {
        // mostly misaligned pieces: shifted bulk copies from the guided queue
        // (parts shrinking to 64 KiB: 6222 against 6036 GB/s for equal 192 KiB
        // parts; the copies whose CTAs sweep the buffers together in small
        // equal parts lose 7-11% with guided parts)
        t.path = kPathBulk;
        t.ctas_per_sm = 1;
        t.stages = 4;
        t.chunk_bytes = 32 * 1024;
        t.schedule = kSchedQueueGuided;
        t.interleave_bytes = 64 * 1024;
      } else if (coll == kAllToAll && S >= 16 * MiB) {
        // bulk ring of 5 slots fed from the shared queue in 64 KiB parts
        t.path = kPathBulk;
        t.ctas_per_sm = 1;
        t.stages = 5;
        t.chunk_bytes = 32 * 1024;
        t.schedule = kSchedQueue;
        t.interleave_bytes = 64 * 1024;
      } else {
        t.unroll = 2;
        t.store_hint = 2;
        if (S >= 1 * MiB && coll == kAllToAll) {
          // working sets of 16-256 MiB: write-back stores keep the outputs in
          // the L2 (a CUDA graph of 10 calls after an L2-sized write: 12.2
          // against 15.0 us at 4 MiB, 21.0 against 25.0 at 8 MiB; at 1 MiB
          // with 4 vectors in flight, 4.96 against 6.22 us)
          t.store_hint = 1;
          if (S < 2 * MiB) t.unroll = 4;
        }
        if (S >= 1 * MiB) {
          t.threads = 512;
          t.min_cta_bytes = 32 * 1024;
        } else if (S >= 128 * KiB) {
          t.min_cta_bytes = 8 * 1024;
        } else if (S >= 32 * KiB) {
          t.min_cta_bytes = 2 * 1024;
        } else {
          t.min_cta_bytes = 128;  // tiny chunks: one piece per CTA
        }
      }
      break;
  }
  return t;
}

Tune tune_merge(const Tune& b, const Tune& o) {
  Tune t = b;
  if (o.layout) t.layout = o.layout;
  if (o.ctas_per_sm) t.ctas_per_sm = o.ctas_per_sm;
  if (o.threads) t.threads = o.threads;
  if (o.unroll) t.unroll = o.unroll;
  if (o.path) t.path = o.path;
  if (o.chunk_bytes) t.chunk_bytes = o.chunk_bytes;
  if (o.stages) t.stages = o.stages;
  if (o.store_hint) t.store_hint = o.store_hint;
  if (o.min_cta_bytes) t.min_cta_bytes = o.min_cta_bytes;
  if (o.interleave_bytes) t.interleave_bytes = o.interleave_bytes;
  if (o.max_ctas) t.max_ctas = o.max_ctas;
  if (o.schedule) t.schedule = o.schedule;
  if (o.snac_lag) t.snac_lag = o.snac_lag;
  return t;
}

Tune resolve_tune(int coll, int table_coll, int world, int dtype, uint64_t bytes_per_rank, const Tune& over) {
  Tune t = tune_merge(tune_table(table_coll, world, dtype, bytes_per_rank), over);
  if (coll == kAllReduce && (t.layout == kTwoShot || t.layout == kTwoShotFused || t.layout == kRing)) {
    // the SNAC layouts' own best (512 threads, two CTAs per SM, no grid cap)
    // unless the caller set these fields; the ring's
    // reduce items have two sources, so two vectors of each in flight
    if (!over.threads) t.threads = 512;
    if (!over.ctas_per_sm) t.ctas_per_sm = 2;
    // two-shot on the register path: the L2 priorities of store_hint 3 (8 x 64
    // MiB bf16: 182 against 186 us write-back, DRAM reads 1.04 against 1.11
    // times the algorithmic bytes)
    if (!over.store_hint)
      t.store_hint = ((t.layout == kTwoShot || t.layout == kTwoShotFused) && t.path == kPathRegister) ? 3 : 1;
    if (!over.max_ctas) t.max_ctas = 0;
    if (t.layout == kRing && !over.unroll) t.unroll = 2;
    if (t.layout == kRing) {
      // ring: tiles of 64 KiB (8 ranks, back to back, stages one wave apart:
      // 404.9 against 444.9 us for 128 KiB at 8 x 64 MiB)
      if (!over.chunk_bytes) t.chunk_bytes = 64 * 1024;
    }
  }
  return t;
}

static int validate_tune(const Tune& t) {
  if (t.layout < kOneShot || t.layout > kTwoShotFused) return PL_ERR_UNSUPPORTED;
  if (t.threads < 64 || t.threads > 512 || t.threads % 32) return PL_ERR_INVALID_ARG;
  if (t.ctas_per_sm < 1 || t.ctas_per_sm > 32) return PL_ERR_INVALID_ARG;
  if (t.unroll < 1 || t.unroll > 8) return PL_ERR_INVALID_ARG;
  if (t.path != kPathRegister && t.path != kPathBulk) return PL_ERR_UNSUPPORTED;
  if (t.chunk_bytes < 1024 || t.chunk_bytes > (64 << 20) || t.chunk_bytes % 16) return PL_ERR_INVALID_ARG;
  if (t.stages < 2 || t.stages > 8) return PL_ERR_INVALID_ARG;
  if (t.store_hint < 1 || t.store_hint > 3) return PL_ERR_INVALID_ARG;
  if (t.min_cta_bytes < 16) return PL_ERR_INVALID_ARG;
  if (t.interleave_bytes < -1 || (t.interleave_bytes > 0 && (t.interleave_bytes < 512 || t.interleave_bytes % 512)))
    return PL_ERR_INVALID_ARG;
  if (t.max_ctas < 0) return PL_ERR_INVALID_ARG;
  if (t.schedule < kSchedItem || t.schedule > kSchedQueueGuided) return PL_ERR_INVALID_ARG;
  if (t.snac_lag < 1 || t.snac_lag > 64) return PL_ERR_INVALID_ARG;
  return PL_OK;
}

int build_plan(int coll, int world, int dtype, const uint64_t* sizes, size_t nsizes,
               const uint8_t* src_res, const uint8_t* dst_res, int sm_count, int max_ctas_per_sm,
               const Tune& tune_in, Plan* out) {
  if (!out || !sizes) return PL_ERR_INVALID_ARG;
  if (world < 1 || world > kMaxWorld) return PL_ERR_INVALID_ARG;
  if (coll < kAllReduce || coll > kAtomReduce) return PL_ERR_UNSUPPORTED;
  if (dtype < kU8 || dtype > kBF16) return PL_ERR_UNSUPPORTED;
  if (sm_count < 1) return PL_ERR_INVALID_ARG;
  if (nsizes != n_sizes(coll, world)) return PL_ERR_INVALID_ARG;
  const bool red = is_reduce_coll(coll);
  if (red && dtype == kU8) return PL_ERR_UNSUPPORTED;

  uint8_t zeros[kMaxWorld] = {};
  if (!src_res) src_res = zeros;
  if (!dst_res) dst_res = zeros;

  Plan p;
  p.coll = coll;
  p.world = world;
  p.dtype = dtype;
  p.elem = red ? elem_size(dtype) : 1;
  const uint64_t E = (uint64_t)p.elem;
  uint64_t per_rank = sizes[0];
  if (coll == kAllGatherV || coll == kAllToAllV || coll == kReduceScatterV) {
    uint64_t total = 0;
    for (size_t i = 0; i < nsizes; ++i) total += sizes[i];
    per_rank = total / (uint64_t)world;
  }
  // A reduce Atom with one destination moves ReduceScatter-shaped traffic
  // (N reads per write); with several it is AllReduce-shaped.
  const int table_coll = (coll == kAtomReduce && nsizes == 3 && sizes[2] == 1) ? (int)kReduceScatter : coll;
  p.tune = resolve_tune(coll, table_coll, world, dtype, per_rank, tune_in);
  if (int st = validate_tune(p.tune)) return st;
  if (p.tune.interleave_bytes < 0) p.tune.interleave_bytes = 0;  // -1 in an override: contiguous shares
  if (max_ctas_per_sm > 0) p.tune.ctas_per_sm = std::min(p.tune.ctas_per_sm, max_ctas_per_sm);

  const uint32_t ALL = all_ranks(world);
  std::vector<Piece> pieces;
  bool sync = false;
  uint32_t n_flags = 0;

  // ------------------------------------------------------------ layouts
  switch (coll) {
    case kAllReduce: {
      const uint64_t S = sizes[0];
      if (S % E) return PL_ERR_ALIGNMENT;
      for (int r = 0; r < world; ++r) p.in_bytes[r] = p.out_bytes[r] = S;
      p.work_bytes = 2ull * world * S;
      p.reduce = true;
      p.nsrc = world;
      if ((p.tune.layout == kTwoShot || p.tune.layout == kTwoShotFused) && world > 1) {
        sync = true;
        const uint64_t n = S / E;
        const uint64_t T = std::max<uint64_t>(16, (uint64_t)p.tune.chunk_bytes / 16 * 16);
        uint64_t start[kMaxWorld + 1];
        start[0] = 0;
        for (int o = 0; o < world; ++o)
          start[o + 1] = start[o] + (n / world + ((uint64_t)o < n % world ? 1 : 0)) * E;
        uint64_t tiles[kMaxWorld], tmax = 0;
        for (int o = 0; o < world; ++o) {
          tiles[o] = ceil_div(start[o + 1] - start[o], T);
          tmax = std::max(tmax, tiles[o]);
        }
        n_flags = (uint32_t)(world * tmax);
        uint64_t n_items = 0;
        for (int o = 0; o < world; ++o) n_items += 2 * tiles[o];
        uint64_t gcap = (uint64_t)p.tune.ctas_per_sm * sm_count;
        if (p.tune.max_ctas > 0) gcap = std::min<uint64_t>(gcap, (uint64_t)p.tune.max_ctas);
        const uint64_t G = std::max<uint64_t>(1, std::min<uint64_t>(gcap, n_items));
        auto reduce_piece = [&](int o, uint64_t t) {
          uint64_t off = start[o] + t * T, len = std::min(T, start[o + 1] - off);
          Piece q{off, off, len, ALL, 1u << o, 0, (uint32_t)(o * tmax + t + 1)};
          push_grouped(pieces, q, dst_res);
        };
        auto copy_piece = [&](int o, uint64_t t) {
          uint64_t off = start[o] + t * T, len = std::min(T, start[o + 1] - off);
          Piece q{off, off, len, 1u << (16 + o), ALL & ~(1u << o), (uint32_t)(o * tmax + t + 1), 0};
          push_grouped(pieces, q, dst_res);
        };
        // Order of the items (the CTAs run item i on CTA i % G, or take them
        // from the shared queue in this order).  Reduce and copy items
        // alternate in a checkerboard of (wave i / G, CTA i % G): every CTA
        // alternates the two kinds and every wave holds about as many of
        // each.  (Rounds of world reduces then world copies gave each CTA one
        // kind whenever G is a multiple of 2 world: at 8 x 64 MiB the reduce
        // CTAs set the pace while the copy CTAs spent 11% of the time
        // waiting.)  A tile's copy comes at least snac_lag x G / 2 positions
        // after its reduce (two waves by default: the reduce has finished by
        // then); a copy that is due but not yet allowed gives its position to
        // the next reduce.
        std::vector<std::pair<int, uint64_t>> tile_order;  // (owner, tile), tile-major
        for (uint64_t t = 0; t < tmax; ++t)
          for (int o = 0; o < world; ++o)
            if (t < tiles[o]) tile_order.emplace_back(o, t);
        const uint64_t nr = tile_order.size();
        const uint64_t D = std::max<uint64_t>(1, (uint64_t)p.tune.snac_lag * G / 2);
        std::vector<uint64_t> rpos(nr);
        uint64_t r = 0, c = 0;
        if (p.tune.layout == kTwoShotFused) {
          if (p.tune.store_hint != 3 || p.tune.schedule != kSchedItem || p.tune.path != kPathRegister)
            return PL_ERR_UNSUPPORTED;  // the L2 kernel kind runs fused items, one CTA sequence each
          // Fused order (the L2 kernel kind): after a first wave of reduces,
          // each item reduces the next tile and, in the same pass, copies the
          // tile reduced D + 1 places earlier -- by the next CTA back, one
          // wave ago (its flag is the item's wait).  Every CTA then streams 8
          // reads and 8 writes per vector, the mix of the one-shot layout,
          // while the copies still consume what other CTAs produced.  Tiles
          // of unequal length (an owner's last), or whose copy destinations
          // sit at different addresses modulo 16, go as separate items.
          auto tile = [&](uint64_t k, uint64_t& off, uint64_t& len) {
            const int o = tile_order[k].first;
            off = start[o] + tile_order[k].second * T;
            len = std::min(T, start[o + 1] - off);
            return o;
          };
          while (r < nr || c < nr) {
            const uint64_t pos = pieces.size();
            const bool can_c = c < r && rpos[c] + D + 1 <= pos;
            uint64_t oa = 0, la = 0, ob = 0, lb = 0;
            int a_own = r < nr ? tile(r, oa, la) : 0;
            int b_own = c < nr ? tile(c, ob, lb) : 0;
            bool coaligned = true;
            for (int d = 0; d < world; ++d)
              if (d != b_own && ((dst_res[d] + ob) & 15u) != ((dst_res[b_own == 0 ? 1 : 0] + ob) & 15u)) coaligned = false;
            if (can_c && r < nr && la == lb && coaligned) {
              rpos[r] = pos;
              pieces.push_back(Piece{oa, ob, la, ALL | (1u << (16 + b_own)), (1u << a_own) | kFused,
                                     (uint32_t)(b_own * tmax + tile_order[c].second + 1),
                                     (uint32_t)(a_own * tmax + tile_order[r].second + 1)});
              ++r;
              ++c;
            } else if (r < nr && !can_c) {
              rpos[r] = pos;
              reduce_piece(tile_order[r].first, tile_order[r].second);
              ++r;
            } else {
              copy_piece(tile_order[c].first, tile_order[c].second);
              ++c;
            }
          }
        } else
        while (r < nr || c < nr) {
          const uint64_t pos = pieces.size();
          const bool want_r = (((pos / G) + (pos % G)) & 1u) == 0;
          const bool can_r = r < nr, can_c = c < r && rpos[c] + D <= pos;
          const bool do_r = can_r && (want_r || !can_c);
          if (do_r) {
            rpos[r] = pos;
            reduce_piece(tile_order[r].first, tile_order[r].second);
            ++r;
          } else {
            copy_piece(tile_order[c].first, tile_order[c].second);
            ++c;
          }
        }
      } else if (p.tune.layout == kRing && world > 1) {
        // Ring (Iris docs, "Device Context", all_reduce_ring: a running sum
        // handed from rank to rank, then the finished data passed around the
        // ring).  The range is cut into `world` chunks and each chunk into
        // tiles (the chunks only order the tiles).  A tile passes through
        // 2 (world - 1) stages, each waiting for the previous one's flag.
        // Reduce stage k = 1 .. world-1 adds rank k's input to the running
        // sum (stage 1: rank 0's input plus rank 1's), so every tile is
        // folded in ascending rank order from rank 0, in binary32, with one
        // rounding at the end: the ascending fold, bit for bit.  The sum
        // lives in the outputs between stages: fp32 in rank k's output; bf16
        // as two 16-bit halves (kSplitDst), low half in rank k - 1's output,
        // high half in rank k's.  The last reduce stage stores the rounded
        // value to rank world-1's output.  Gather stage m = 1 .. world-1
        // copies the output of rank world-2+m (mod world) to rank
        // world-1+m (mod world).  Every output byte is written more than once
        // (the sum first, the result last) and each overwrite waits, through
        // the chain, for the read of what it replaces.
        if (p.tune.path != kPathRegister) return PL_ERR_UNSUPPORTED;  // the register-path kernel only
        sync = true;
        p.nsrc = 2;
        const bool split = dtype == kBF16;
        const uint64_t n = S / E;
        const uint64_t T = std::max<uint64_t>(16, (uint64_t)p.tune.chunk_bytes / 16 * 16);
        uint64_t start[kMaxWorld + 1];
        start[0] = 0;
        for (int j = 0; j < world; ++j)
          start[j + 1] = start[j] + (n / world + ((uint64_t)j < n % world ? 1 : 0)) * E;
        uint64_t tiles[kMaxWorld], tmax = 0, n_items = 0;
        const uint32_t stages = 2u * (uint32_t)world - 2u;
        for (int j = 0; j < world; ++j) {
          tiles[j] = ceil_div(start[j + 1] - start[j], T);
          tmax = std::max(tmax, tiles[j]);
          n_items += tiles[j] * stages;
        }
        // one flag per (chunk, tile, stage) except each tile's last stage
        n_flags = (uint32_t)((uint64_t)world * tmax * (stages - 1));
        auto flag = [&](int j, uint64_t t, uint32_t st) {
          return (uint32_t)(((uint64_t)j * tmax + t) * (stages - 1) + st + 1);
        };
        const uint64_t gcap = (uint64_t)p.tune.ctas_per_sm * sm_count;
        const uint64_t G = std::max<uint64_t>(1, std::min<uint64_t>(gcap, n_items));
        // A tile's stage comes at least D = snac_lag x G / 2 places (one
        // wave of CTAs by default) after its previous stage in the items'
        // order: the previous stage has usually finished, and the running
        // sum is read back while it is still in the L2.
        const uint64_t D = std::max<uint64_t>(1, (uint64_t)p.tune.snac_lag * G / 2);
        auto stage_piece = [&](int j, uint64_t t, uint32_t st) {
          const uint64_t off = start[j] + t * T, len = std::min(T, start[j + 1] - off);
          uint32_t src, dst;
          if (st + 1 < (uint32_t)world) {
            const int k = (int)st + 1;
            const bool last = k == world - 1;
            if (k == 1)
              src = 1u | 2u;                                  // rank 0's input + rank 1's
            else if (split)
              src = (1u << k) | (3u << (16 + k - 2));         // rank k's input + halves in outputs k-2, k-1
            else
              src = (1u << k) | (1u << (16 + k - 1));         // rank k's input + the sum in output k-1
            dst = (last || !split) ? (1u << k) : (3u << (k - 1));
            if (split && k > 1) dst |= kSplitSrc;
            if (split && !last) dst |= kSplitDst;
          } else {
            const int m = (int)st - (world - 1) + 1;
            src = 1u << (16 + (world - 2 + m) % world);
            dst = 1u << ((world - 1 + m) % world);
          }
          Piece q{off, off, len, src, dst, st ? flag(j, t, st - 1) : 0u, st + 1 < stages ? flag(j, t, st) : 0u};
          if (dst & (kSplitSrc | kSplitDst)) {
            if (q.len) pieces.push_back(q);  // one item: the halves are two values, not copies of one
          } else {
            push_grouped(pieces, q, dst_res);
          }
        };
        // Emission: at every place, the oldest pending stage if it is due,
        // else the first stage of the next tile (tile-major over the chunks),
        // else the oldest pending stage anyway (it will wait for its flag).
        // Stages become due in the order they were queued, so a FIFO holds
        // them in due order.
        struct Pending {
          uint64_t due;
          int j;
          uint64_t t;
          uint32_t st;
        };
        std::vector<Pending> fifo;
        size_t head = 0;
        uint64_t next_t = 0;
        int next_j = 0;
        auto advance_new = [&]() {  // the next (chunk, tile) that exists
          while (next_t < tmax && (uint64_t)tiles[next_j] <= next_t) {
            if (++next_j == world) {
              next_j = 0;
              ++next_t;
            }
          }
        };
        advance_new();
        while (head < fifo.size() || next_t < tmax) {
          const uint64_t pos = pieces.size();
          Pending e;
          if (head < fifo.size() && (fifo[head].due <= pos || next_t >= tmax)) {
            e = fifo[head++];
          } else {
            e = Pending{0, next_j, next_t, 0};
            if (++next_j == world) {
              next_j = 0;
              ++next_t;
            }
            advance_new();
          }
          stage_piece(e.j, e.t, e.st);
          if (e.st + 1 < stages) fifo.push_back(Pending{pieces.size() - 1 + D, e.j, e.t, e.st + 1});
        }
      } else {
        // one rank: every layout is the one-shot copy (and the two-shot's L2
        // priorities have no copies to serve)
        if ((p.tune.layout == kTwoShot || p.tune.layout == kTwoShotFused) && p.tune.store_hint == 3) p.tune.store_hint = 1;
        p.tune.layout = kOneShot;
        push_grouped(pieces, Piece{0, 0, S, ALL, ALL, 0, 0}, dst_res);
      }
      break;
    }
    case kReduceScatter: {
      const uint64_t S = sizes[0];
      if (S % E) return PL_ERR_ALIGNMENT;
      if ((S / E) % world) return PL_ERR_INVALID_ARG;
      const uint64_t c = S / world;
      for (int r = 0; r < world; ++r) {
        p.in_bytes[r] = S;
        p.out_bytes[r] = c;
        push_grouped(pieces, Piece{r * c, 0, c, ALL, 1u << r, 0, 0}, dst_res);
      }
      p.work_bytes = (uint64_t)world * S + S;
      p.reduce = true;
      p.nsrc = world;
      break;
    }
    case kReduceScatterV: {
      uint64_t total = 0;
      for (int r = 0; r < world; ++r) {
        if (sizes[r] % E) return PL_ERR_ALIGNMENT;
        total += sizes[r];
      }
      uint64_t off = 0;
      for (int r = 0; r < world; ++r) {
        p.in_bytes[r] = total;
        p.out_bytes[r] = sizes[r];
        push_grouped(pieces, Piece{off, 0, sizes[r], ALL, 1u << r, 0, 0}, dst_res);
        off += sizes[r];
      }
      p.work_bytes = (uint64_t)world * total + total;
      p.reduce = true;
      p.nsrc = world;
      break;
    }
    case kAllGather: {
      const uint64_t S = sizes[0];
      for (int s = 0; s < world; ++s) {
        p.in_bytes[s] = S;
        p.out_bytes[s] = (uint64_t)world * S;
        push_grouped(pieces, Piece{0, s * S, S, 1u << s, ALL, 0, 0}, dst_res);
      }
      p.work_bytes = (uint64_t)world * S + (uint64_t)world * world * S;
      break;
    }
    case kAllToAll: {
      const uint64_t S = sizes[0];
      if (S % world) return PL_ERR_INVALID_ARG;
      const uint64_t c = S / world;
      for (int s = 0; s < world; ++s) p.in_bytes[s] = p.out_bytes[s] = S;
      for (int s = 0; s < world; ++s)
        for (int d = 0; d < world; ++d)
          push_grouped(pieces, Piece{d * c, s * c, c, 1u << s, 1u << d, 0, 0}, dst_res);
      p.work_bytes = 2ull * world * S;
      break;
    }
    case kAllGatherV: {
      uint64_t total = 0;
      for (int s = 0; s < world; ++s) total += sizes[s];
      uint64_t displ = 0;
      for (int s = 0; s < world; ++s) {
        p.in_bytes[s] = sizes[s];
        p.out_bytes[s] = total;
        push_grouped(pieces, Piece{0, displ, sizes[s], 1u << s, ALL, 0, 0}, dst_res);
        displ += sizes[s];
      }
      p.work_bytes = total + (uint64_t)world * total;
      break;
    }
    case kAllToAllV: {
      uint64_t total = 0;
      for (int s = 0; s < world; ++s) {
        uint64_t send = 0;
        for (int d = 0; d < world; ++d) send += sizes[s * world + d];
        p.in_bytes[s] = send;
        total += send;
      }
      for (int d = 0; d < world; ++d) {
        uint64_t recv = 0;
        for (int s = 0; s < world; ++s) recv += sizes[s * world + d];
        p.out_bytes[d] = recv;
      }
      for (int s = 0; s < world; ++s) {
        for (int d = 0; d < world; ++d) {
          uint64_t sdispl = 0, rdispl = 0;
          for (int k = 0; k < d; ++k) sdispl += sizes[s * world + k];
          for (int k = 0; k < s; ++k) rdispl += sizes[k * world + d];
          push_grouped(pieces, Piece{sdispl, rdispl, sizes[s * world + d], 1u << s, 1u << d, 0, 0},
                       dst_res);
        }
      }
      p.work_bytes = 2ull * total;
      break;
    }
    case kAtomCopy: {
      const uint64_t S = sizes[0];
      p.in_bytes[0] = S;
      for (int d = 0; d < world; ++d) p.out_bytes[d] = S;
      push_grouped(pieces, Piece{0, 0, S, 1u, ALL, 0, 0}, dst_res);
      p.work_bytes = S + (uint64_t)world * S;
      break;
    }
    case kAtomReduce: {
      const uint64_t S = sizes[0];
      const uint64_t ns = sizes[1], nd = sizes[2];
      if (ns < 1 || nd < 1 || ns > (uint64_t)world || nd > (uint64_t)world) return PL_ERR_INVALID_ARG;
      if (S % E) return PL_ERR_ALIGNMENT;
      for (uint64_t s = 0; s < ns; ++s) p.in_bytes[s] = S;
      for (uint64_t d = 0; d < nd; ++d) p.out_bytes[d] = S;
      push_grouped(pieces, Piece{0, 0, S, all_ranks((int)ns), all_ranks((int)nd), 0, 0}, dst_res);
      p.work_bytes = (ns + nd) * S;
      p.reduce = ns > 1;
      p.nsrc = (int)ns;
      break;
    }
  }
  // store_hint 3 keeps reduce results evict-last in the L2 until a copy has
  // read them back: only the two-shot layout (register path) has such copies
  if (p.tune.store_hint == 3 &&
      !(coll == kAllReduce && (p.tune.layout == kTwoShot || p.tune.layout == kTwoShotFused) && sync &&
        p.tune.path == kPathRegister))
    return PL_ERR_INVALID_ARG;
  if (!p.reduce) p.nsrc = 1;
  // the register-path kernel for more than 8 sources is built for CTAs of at
  // most 256 threads (room for 128 registers)
  if (p.tune.path == kPathRegister && p.nsrc > 8) p.tune.threads = std::min(p.tune.threads, 256);
  // Streamed schedules are copy plans on the bulk path.  The shared queue
  // serves every plan on the register path, and copy plans on the bulk path.
  if (p.tune.schedule == kSchedStream && (p.reduce || sync || p.tune.path != kPathBulk)) return PL_ERR_UNSUPPORTED;
  if ((p.tune.schedule == kSchedQueue || p.tune.schedule == kSchedQueueGuided) && p.tune.path == kPathBulk &&
      (p.reduce || sync))
    return PL_ERR_UNSUPPORTED;

  // ------------------------------------------------------------ tiling
  uint64_t gcap = (uint64_t)p.tune.ctas_per_sm * (uint64_t)sm_count;
  if (p.tune.max_ctas > 0) gcap = std::min<uint64_t>(gcap, (uint64_t)p.tune.max_ctas);
  if (sync) {
    p.strided = true;
    p.sync = true;
    p.queue = p.tune.schedule == kSchedQueue || p.tune.schedule == kSchedQueueGuided;
    p.n_flags = (int)n_flags;
    const uint64_t n = pieces.size();
    p.grid = (int)std::max<uint64_t>(1, std::min<uint64_t>(gcap, n));
    p.items.reserve(n);
    for (const Piece& q : pieces)
      p.items.push_back(Item{q.src_off, q.dst_off, q.len, q.src_mask, q.dst_mask, q.wait, q.notify});
  } else {
    // The concatenated piece space is cut into `nparts` near-equal parts at
    // 512-byte granules of each piece.  Without interleaving nparts = grid and
    // CTA c takes part c (one contiguous share).  With interleave_bytes = T,
    // nparts = k * grid with parts of about T bytes, and CTA c takes parts
    // c, c + grid, c + 2 grid, ... in that order: at any moment the CTAs work
    // on neighbouring parts, and every CTA still gets the same number of bytes.
    // The queue schedule cuts the same parts (of interleave_bytes, else about
    // kQueuePartBytes) but keeps them in one list in global order; CTAs take
    // the next item from a shared counter, so faster CTAs take more.
    uint64_t W = 0;
    for (const Piece& q : pieces) W += q.len;
    uint64_t G = std::max<uint64_t>(1, std::min<uint64_t>(gcap, ceil_div(W, (uint64_t)p.tune.min_cta_bytes)));
    // shares of at least one 512-byte granule, except that pieces smaller than
    // that may each get a CTA of their own (latency of small calls)
    G = std::min<uint64_t>(G, std::max<uint64_t>({1, W / kSplitGranule, (uint64_t)pieces.size()}));
    const bool queue = p.tune.schedule == kSchedQueue || p.tune.schedule == kSchedQueueGuided;
    // part ends in the concatenated piece space (the last one is W)
    std::vector<uint64_t> ends;
    if (p.tune.schedule == kSchedQueueGuided) {
      // guided: each part is 1/(2 grid) of what is left, between
      // interleave_bytes and four times that: larger parts first (fewer
      // items), small ones last (the CTAs that run slower stop at nearly the
      // same time).  The cap keeps the CTAs' first parts close together in
      // the buffers (AllToAllV workload: 86.8 against 88.9 us uncapped)
      const uint64_t T = p.tune.interleave_bytes > 0 ? (uint64_t)p.tune.interleave_bytes : kQueuePartBytes;
      uint64_t pos = 0;
      while (pos < W) {
        uint64_t part = std::max<uint64_t>(T, std::min<uint64_t>(4 * T, (W - pos) / (2 * G)));
        part = (part + kSplitGranule - 1) & ~(kSplitGranule - 1);
        pos = (W - pos <= part) ? W : pos + part;
        ends.push_back(pos);
      }
    } else {
      uint64_t k = 1;
      if (p.tune.interleave_bytes > 0 || queue) {
        const uint64_t T = p.tune.interleave_bytes > 0 ? (uint64_t)p.tune.interleave_bytes : kQueuePartBytes;
        k = std::max<uint64_t>(1, (W + T * G / 2) / (T * G));
        k = std::min<uint64_t>(k, std::max<uint64_t>(1, W / (kSplitGranule * G)));
      }
      const uint64_t n = k * G;
      for (uint64_t j = 0; j < n; ++j)
        // exact integer part boundary: floor((j+1) * W / n) without overflow
        ends.push_back(j + 1 == n ? W : (uint64_t)(((unsigned __int128)(j + 1) * W) / n));
    }
    const uint64_t nparts = ends.size();
    p.queue = queue;
    p.grid = (int)G;
    std::vector<uint64_t> start(pieces.size() + 1, 0);
    for (size_t i = 0; i < pieces.size(); ++i) start[i + 1] = start[i] + pieces[i].len;
    // boundary b of the concatenated space -> (piece, offset rounded down to the granule)
    auto locate = [&](uint64_t b, size_t& pi, uint64_t& off) {
      if (b >= W) {
        pi = pieces.size();
        off = 0;
        return;
      }
      pi = (size_t)(std::upper_bound(start.begin(), start.end(), b) - start.begin()) - 1;
      off = (b - start[pi]) & ~(kSplitGranule - 1);
    };
    std::vector<std::vector<Item>> per_cta((size_t)G);
    size_t cp = 0;
    uint64_t co = 0;
    for (uint64_t j = 0; j < nparts; ++j) {
      size_t ep;
      uint64_t eo;
      if (j + 1 == nparts) {
        ep = pieces.size();
        eo = 0;
      } else {
        locate(ends[j], ep, eo);
      }
      // the shared queue hands out items in global order: one list
      std::vector<Item>& dst = per_cta[queue ? 0 : (size_t)(j % G)];
      while (cp < ep || (cp == ep && co < eo)) {
        const Piece& q = pieces[cp];
        const uint64_t end = (cp == ep) ? eo : q.len;
        // items stay below 1 GiB so the Atoms can count 16-byte vectors in 32 bits
        for (uint64_t a = co; a < end; a += kMaxItemBytes) {
          const uint64_t l = std::min<uint64_t>(kMaxItemBytes, end - a);
          dst.push_back(Item{q.src_off + a, q.dst_off + a, l, q.src_mask, q.dst_mask, 0, 0});
        }
        if (cp == ep) {
          co = eo;
          break;
        }
        ++cp;
        co = 0;
      }
    }
    p.cta_begin.push_back(0);
    for (const auto& v : per_cta) {
      p.items.insert(p.items.end(), v.begin(), v.end());
      p.cta_begin.push_back((uint32_t)p.items.size());
    }
  }
  *out = std::move(p);
  return PL_OK;
}

std::string check_plan(const Plan& p) {
  std::ostringstream err;
  const uint32_t ALL = all_ranks(p.world);
  std::vector<int64_t> notified_at(p.n_flags, -1);
  for (size_t i = 0; i < p.items.size(); ++i) {
    const Item& it = p.items[i];
    if (it.notify) {
      if (it.notify > (uint32_t)p.n_flags) return "notify flag out of range";
      notified_at[it.notify - 1] = (int64_t)i;
    }
  }
  // accesses to every output: {lo, hi, item, is_write}
  struct Acc {
    uint64_t lo, hi;
    int64_t item;
    bool write;
  };
  std::vector<std::vector<Acc>> acc(p.world);
  for (size_t i = 0; i < p.items.size(); ++i) {
    const Item& it = p.items[i];
    if (it.len == 0) return "empty item";
    const uint32_t in_bits = it.src_mask & 0xFFFFu, out_bits = it.src_mask >> 16;
    const uint32_t dst_bits = it.dst_mask & kDstRanks, split = it.dst_mask & (kSplitSrc | kSplitDst);
    const bool fused = (it.dst_mask & kFused) != 0;
    if ((in_bits & ~ALL) || (out_bits & ~ALL)) return "source mask outside the world";
    if (!dst_bits || (dst_bits & ~ALL) || (it.dst_mask & ~(kDstRanks | kSplitSrc | kSplitDst | kFused)))
      return "destination mask empty or outside the world";
    const int nsrc = popcount32(it.src_mask);
    if (nsrc < 1) return "item without a source";
    if (fused) {
      // reduce the tile at src_off into the destination, copy the tile at
      // dst_off from the output source to every other output
      if (p.tune.layout != kTwoShotFused || split || popcount32(out_bits) != 1 || popcount32(dst_bits) != 1 ||
          popcount32(in_bits) < 2 || !it.wait || !it.notify)
        return "a fused item outside the two-shot layout";
      if ((it.src_off | it.dst_off | it.len) % (uint64_t)p.elem) return "reduce not element aligned";
      for (uint32_t m = in_bits; m; m &= m - 1)
        if (it.src_off + it.len > p.in_bytes[__builtin_ctz(m)]) return "a fused item reads past an input";
      const int ob = __builtin_ctz(out_bits), oa = __builtin_ctz(dst_bits);
      if (it.dst_off + it.len > p.out_bytes[ob] || it.src_off + it.len > p.out_bytes[oa])
        return "a fused item reaches past an output";
      acc[oa].push_back({it.src_off, it.src_off + it.len, (int64_t)i, true});
      acc[ob].push_back({it.dst_off, it.dst_off + it.len, (int64_t)i, false});
      for (int d = 0; d < p.world; ++d)
        if (d != ob) {
          if (it.dst_off + it.len > p.out_bytes[d]) return "a fused item writes past an output";
          acc[d].push_back({it.dst_off, it.dst_off + it.len, (int64_t)i, true});
        }
      if (it.wait > (uint32_t)p.n_flags) return "wait flag out of range";
      const int64_t at = notified_at[it.wait - 1];
      if (at < 0) return "wait without a notify";
      if ((p.strided || p.queue) && at >= (int64_t)i) return "wait without an earlier notify";
      continue;
    }
    if (split) {
      // the ring's binary32 running sum over bf16 data: two output halves in
      // neighbouring ranks, read and / or written by one reduce item
      if (p.tune.layout != kRing || p.dtype != kBF16 || nsrc < 2) return "split sum outside the bf16 ring";
      if ((it.dst_mask & kSplitSrc) && (popcount32(out_bits) != 2 || (out_bits & (out_bits >> 1)) == 0))
        return "split source is not two neighbouring outputs";
      if ((it.dst_mask & kSplitDst) && (popcount32(dst_bits) != 2 || (dst_bits & (dst_bits >> 1)) == 0))
        return "split destination is not two neighbouring outputs";
    } else if (nsrc > 1 && popcount32(out_bits) > 1) {
      return "a reduce reads several outputs";
    }
    // a reduce reads an output only in the ring layout (whose kernel loads
    // such sources through the L2) and only after waiting for its producer
    if (nsrc > 1 && out_bits && (p.tune.layout != kRing || !it.wait)) return "a reduce reads outputs";
    if (nsrc > 1 && ((it.src_off | it.dst_off | it.len) % (uint64_t)p.elem)) return "reduce not element aligned";
    for (uint32_t m = in_bits; m; m &= m - 1) {
      int r = __builtin_ctz(m);
      if (it.src_off + it.len > p.in_bytes[r]) {
        err << "item " << i << " reads past input " << r;
        return err.str();
      }
    }
    for (uint32_t m = out_bits; m; m &= m - 1) {
      int r = __builtin_ctz(m);
      if (it.src_off + it.len > p.out_bytes[r]) return "reads past an output";
      acc[r].push_back({it.src_off, it.src_off + it.len, (int64_t)i, false});
    }
    for (uint32_t m = dst_bits; m; m &= m - 1) {
      int r = __builtin_ctz(m);
      if (it.dst_off + it.len > p.out_bytes[r]) {
        err << "item " << i << " writes past output " << r;
        return err.str();
      }
      acc[r].push_back({it.dst_off, it.dst_off + it.len, (int64_t)i, true});
    }
    if (it.wait) {
      if (it.wait > (uint32_t)p.n_flags) return "wait flag out of range";
      const int64_t at = notified_at[it.wait - 1];
      if (at < 0) return "wait without a notify";
      // strided and queued plans: every wait follows its notify in the
      // global order (the queue hands items out in that order)
      if ((p.strided || p.queue) && at >= (int64_t)i) return "wait without an earlier notify";
    }
  }
  if (p.sync && !p.queue) {
    // the CTAs' sequences and the waits must not form a cycle (all CTAs are
    // resident, so then the earliest unfinished item can always run)
    const size_t n = p.items.size();
    std::vector<std::vector<uint32_t>> out(n);
    std::vector<uint32_t> indeg(n, 0);
    auto edge = [&](size_t a, size_t b) {
      out[a].push_back((uint32_t)b);
      ++indeg[b];
    };
    if (p.strided) {
      for (size_t i = 0; i + (size_t)p.grid < n; ++i) edge(i, i + (size_t)p.grid);
    } else {
      if (p.cta_begin.size() != (size_t)p.grid + 1 || p.cta_begin.front() != 0 || p.cta_begin.back() != n)
        return "cta ranges";
      for (size_t c = 0; c + 1 < p.cta_begin.size(); ++c)
        for (uint32_t i = p.cta_begin[c]; i + 1 < p.cta_begin[c + 1]; ++i) edge(i, i + 1);
    }
    for (size_t i = 0; i < n; ++i)
      if (p.items[i].wait) edge((size_t)notified_at[p.items[i].wait - 1], i);
    std::vector<uint32_t> ready;
    for (size_t i = 0; i < n; ++i)
      if (!indeg[i]) ready.push_back((uint32_t)i);
    size_t done = 0;
    while (!ready.empty()) {
      const uint32_t i = ready.back();
      ready.pop_back();
      ++done;
      for (uint32_t j : out[i])
        if (--indeg[j] == 0) ready.push_back(j);
    }
    if (done != n) return "the waits of the plan can deadlock";
  }
  // item b comes after item a through a chain of waits: b waits for a flag
  // that a, or an item after a in that sense, notified
  auto chain_to = [&](int64_t a, int64_t b) {
    int64_t k = b;
    for (size_t hops = 0; hops <= p.items.size(); ++hops) {
      const uint32_t w = p.items[(size_t)k].wait;
      if (!w) return false;
      k = notified_at[w - 1];
      if (k == a) return true;
    }
    return false;
  };
  auto chained = [&](int64_t a, int64_t b) { return chain_to(a, b) || chain_to(b, a); };
  for (int r = 0; r < p.world; ++r) {
    auto& v = acc[r];
    std::sort(v.begin(), v.end(), [](const Acc& x, const Acc& y) {
      return x.lo != y.lo ? x.lo < y.lo : x.hi != y.hi ? x.hi < y.hi : x.item < y.item;
    });
    uint64_t covered = 0, end_any = 0, end_write = 0;
    for (size_t k = 0; k < v.size();) {
      // one group: the accesses to one identical range, in item order
      size_t e = k;
      bool any_write = false;
      while (e < v.size() && v[e].lo == v[k].lo && v[e].hi == v[k].hi) any_write |= v[e++].write;
      if (v[k].lo < end_write || (any_write && v[k].lo < end_any))
        return "an output byte is accessed under partly overlapping ranges, one of them written";
      // every pair with a write must be ordered by a chain of waits
      for (size_t x = k; x < e; ++x)
        for (size_t y = x + 1; y < e; ++y)
          if ((v[x].write || v[y].write) && v[x].item != v[y].item && !chained(v[x].item, v[y].item))
            return v[x].write && v[y].write ? "an output byte is written twice" : "a read and a write of an output are not ordered";
      if (any_write) {
        covered += v[k].hi - v[k].lo;
        end_write = std::max(end_write, v[k].hi);
      }
      end_any = std::max(end_any, v[k].hi);
      k = e;
    }
    if (covered != p.out_bytes[r]) {
      err << "output " << r << " covered " << covered << " of " << p.out_bytes[r];
      return err.str();
    }
  }
  if (!p.strided) {
    if (p.cta_begin.size() != (size_t)p.grid + 1) return "cta ranges";
    for (size_t c = 0; c + 1 < p.cta_begin.size(); ++c)
      if (p.cta_begin[c] > p.cta_begin[c + 1]) return "cta ranges not monotone";
    if (p.cta_begin.front() != 0 || p.cta_begin.back() != p.items.size()) return "cta ranges do not cover";
  }
  return "";
}

}  // namespace pl
