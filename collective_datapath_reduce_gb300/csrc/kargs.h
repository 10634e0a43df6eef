// Kernel arguments of one collective launch, shared by the host runtime and
// the device code.  Passed by value as a __grid_constant__ parameter: the
// per-rank buffer pointers live in the kernel's parameter space, so a plan
// (offsets only) serves any buffers with the same alignment.
#pragma once

#include <stdint.h>

#include "plan.h"

namespace pl {

// Control words at the start of the workspace.
enum : int { kCtlStatus = 0, kCtlEpoch = 1, kCtlDone = 2, kCtlQueue = 3, kCtlQueueDone = 4 };
constexpr int kCtlBytes = 256;   // flags start here
constexpr int kDevTimeout = 7;   // PL_ERR_TIMEOUT
constexpr int kDevBounds = 9;    // PL_ERR_BOUNDS (checking build)

struct KArgs {
  const char* in[kMaxWorld];
  char* out[kMaxWorld];
  const Item* items;
  const uint32_t* cta_begin;  // contiguous assignment (nullptr when strided)
  uint32_t n_items;
  uint32_t strided;           // item i on CTA i % grid (else contiguous ranges)
  uint32_t sync;              // the plan has SNAC flags: epoch, status and done counter in use
  uint32_t queue;             // items are taken from the shared queue counter (streamed copies)
  uint32_t* flags;
  uint32_t* ctl;              // status, epoch, done counter, queue counter, queue done counter
  unsigned long long timeout_ns;
  uint32_t drop_notify;       // 1 + item whose notify is skipped, or 0
  int nsrc;                   // sources of each reduce item
  int store_hint;             // 1 write-back, 2 streaming
  int stages;                 // bulk path: slots in the shared-memory ring
  uint32_t chunk_bytes;       // bulk path: bytes per source tile in a slot
  unsigned long long* trace;  // trace buffer (header word + records), or nullptr
  uint32_t trace_cap;         // records the trace buffer holds
  uint64_t in_bytes[kMaxWorld];   // bytes of each input and output buffer (the
  uint64_t out_bytes[kMaxWorld];  // checking build tests every item against them)
  uint32_t flag_cap;              // flags the workspace holds (cleared when the epoch wraps)
};

// One trace record (32 bytes): which CTA ran which item, when, and how long it
// waited for its SNAC flag.  The buffer starts with one 64-bit record count.
struct TraceRecord {
  unsigned long long t_start;  // %globaltimer when the item was picked up (ns)
  unsigned long long t_end;    // when the CTA had issued the item's stores (and raised its flag)
  uint32_t cta;
  uint32_t item;
  uint32_t wait_ns;            // time in the consume wait
  uint32_t len_kib;            // item length in KiB (rounded down)
};
static_assert(sizeof(TraceRecord) == 32, "trace record layout");

// Kernel entry points (device function addresses), by variant.  nullptr when
// the variant is not built.
const void* kernel_copy(int unroll);
const void* kernel_reduce_f32(int nsrc, int unroll);
const void* kernel_reduce_bf16(int nsrc, int unroll);
// Two-shot AllReduce with L2 priorities (store_hint 3).
const void* kernel_reduce_l2_f32(int nsrc, int unroll);
const void* kernel_reduce_l2_bf16(int nsrc, int unroll);
// Ring AllReduce (reduce items that read running sums stored in the same launch).
const void* kernel_reduce_ring_f32(int unroll);
const void* kernel_reduce_ring_bf16(int unroll);
// TMA bulk pipeline variants (dynamic shared memory).
const void* kernel_bulk_copy();
const void* kernel_bulk_reduce_f32(int nsrc);
const void* kernel_bulk_reduce_bf16(int nsrc);
// Streamed bulk copies (one pipeline across a CTA's items; optional shared queue).
const void* kernel_stream_copy();

}  // namespace pl
