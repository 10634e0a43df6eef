// Plans: the layout of a collective split into per-CTA work items.
//
// A layout (Purlin README, purlin 0.6.4, "Key Idea": layouts describe how
// inputs and outputs are distributed and whether each piece is copied or
// reduced) is a list of pieces.  A piece moves one contiguous byte range:
// it reads the same offset of every source buffer named in its source mask
// (one source = copy Atom, several = N-to-1 reduce Atom, folded in ascending
// mask-bit order) and writes the result to the same offset of every
// destination buffer named in its destination mask.  Tiling cuts the pieces
// into work items and assigns the items to a persistent grid of CTAs.
//
// Host-only code: no CUDA types here, so the same plan can be built and
// checked on a machine without a GPU.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

namespace pl {

constexpr int kMaxWorld = 16;

enum Coll : int {
  kAllReduce = 0,
  kReduceScatter = 1,
  kAllGather = 2,
  kAllToAll = 3,
  kAllGatherV = 4,
  kAllToAllV = 5,
  kReduceScatterV = 6,
  kAtomCopy = 7,
  kAtomReduce = 8,
};

enum Dtype : int { kU8 = 0, kF32 = 1, kBF16 = 2 };

enum Layout : int { kLayoutAuto = 0, kOneShot = 1, kTwoShot = 2, kRing = 3, kTwoShotFused = 4 };

enum Path : int { kPathRegister = 1, kPathBulk = 2 };

// How a CTA walks its work.  Item: one item at a time (each bulk item fills
// and drains its own pipeline).  Stream: a CTA's items flow through one
// continuous bulk pipeline.  Queue: streamed, and the CTAs take items in
// order from a counter shared by the grid instead of fixed shares.  Stream
// and queue serve copy plans on the bulk path.  Guided queue: the queue with
// parts that shrink toward the end of the work.
enum Schedule : int { kSchedItem = 1, kSchedStream = 2, kSchedQueue = 3, kSchedQueueGuided = 4 };

// Device format of one work item (40 bytes).  Same field meanings as
// purlin_item in the public header, minus the CTA bookkeeping.
struct Item {
  uint64_t src_off;
  uint64_t dst_off;
  uint64_t len;
  uint32_t src_mask;  // bit r: input of rank r; bit 16 + r: output of rank r
  uint32_t dst_mask;  // bit r: output of rank r; bits 30, 31: kSplitSrc, kSplitDst
  uint32_t wait;      // 0 or flag index + 1
  uint32_t notify;    // 0 or flag index + 1
};
static_assert(sizeof(Item) == 40, "device item layout");

// Ring AllReduce over bf16 data: the running sum is a binary32 value kept as
// two 16-bit halves in two rank outputs, the low half in the lower-numbered
// rank, the high half in the higher-numbered one.  kSplitSrc: the item's two
// output sources are those halves (its input sources are added to the sum
// they form).  kSplitDst: its two destinations receive the halves of the new
// sum instead of a rounded bf16 value.  Only the ring kernel reads them.
constexpr uint32_t kSplitSrc = 1u << 30;
constexpr uint32_t kSplitDst = 1u << 31;
// Two-shot AllReduce with L2 priorities: one item reduces the tile at src_off
// (sources: the item's input bits; destination: its one destination bit) and,
// in the same pass, copies the tile at dst_off from the output named by its
// output source bit to every other rank's output.  It notifies the flag of
// the tile it reduces and waits for the flag of the tile it copies.
constexpr uint32_t kFused = 1u << 29;
constexpr uint32_t kDstRanks = 0xFFFFu;

struct Tune {
  int layout = 0;
  int ctas_per_sm = 0;
  int threads = 0;
  int unroll = 0;
  int path = 0;
  int chunk_bytes = 0;
  int stages = 0;
  int store_hint = 0;
  int min_cta_bytes = 0;
  int interleave_bytes = 0;  // > 0: parts of about this size, CTA c takes parts c, c + grid, ...
  int max_ctas = 0;          // > 0: cap on the grid size
  int schedule = 0;          // Schedule
  int snac_lag = 0;          // two-shot: positions between a tile's reduce and its copies, in half waves
};

struct Plan {
  int coll = 0, world = 0, dtype = 0, elem = 1;
  bool reduce = false;       // items with several sources exist
  int nsrc = 1;              // sources of each reduce item
  Tune tune;                 // resolved tuning (no zero fields)
  std::vector<Item> items;   // global order
  std::vector<uint32_t> cta_begin;  // contiguous assignment: grid + 1 entries
  bool strided = false;      // item i runs on CTA i % grid, in increasing i
  bool sync = false;         // items wait on / notify SNAC flags (CTAs must be co-resident)
  bool queue = false;        // CTAs take items from the shared queue (items in global order)
  int grid = 0;
  int n_flags = 0;           // SNAC flags used (two-shot and ring layouts)
  uint64_t in_bytes[kMaxWorld] = {};   // bytes each input must hold
  uint64_t out_bytes[kMaxWorld] = {};  // bytes each output must hold
  uint64_t work_bytes = 0;   // algorithmic bytes (each input byte read once, each output byte written once)
};

// Sizes argument of a collective, as in purlin_plan_describe.
struct Sizes {
  std::vector<uint64_t> v;
};

int elem_size(int dtype);

// Tuning table entry for a call, before overrides.
Tune tune_table(int coll, int world, int dtype, uint64_t bytes_per_rank);
// Fill zero fields of `over` from `base`.
Tune tune_merge(const Tune& base, const Tune& over);
// The tuning a call runs with: the table entry (of `table_coll`), then the
// override, then the layout's own defaults (two-shot AllReduce).  The plan
// may still cap the thread count (more than 8 sources on the register path)
// and the CTAs per SM (co-residency of SNAC plans).
Tune resolve_tune(int coll, int table_coll, int world, int dtype, uint64_t bytes_per_rank, const Tune& over);

// Build the plan.  src_res / dst_res: address of each rank's buffer modulo 16
// (world entries).  max_ctas_per_sm caps tune.ctas_per_sm (residency limit
// for plans whose CTAs wait on each other).  Returns 0 or a purlin_status.
int build_plan(int coll, int world, int dtype, const uint64_t* sizes, size_t nsizes,
               const uint8_t* src_res, const uint8_t* dst_res, int sm_count,
               int max_ctas_per_sm, const Tune& tune, Plan* out);

// Check a plan: every item inside the buffers it names, masks inside the
// world, flags in range, each wait after its notify in global order, every
// output byte written, and two accesses to one output byte, one of them a
// write, only on identical ranges linked by a chain of waits.
// Returns an empty string when the plan is sound, else a description.
std::string check_plan(const Plan& p);

// Number of sizes the collective takes for `world` ranks.
size_t n_sizes(int coll, int world);

}  // namespace pl
