// Streamed TMA copies: every copy item of a CTA flows through one continuous
// bulk pipeline, and the CTA can take its items from a queue shared by the
// whole grid.
//
// The item-at-a-time bulk kernel (kernels_bulk.cuh) fills its shared-memory
// ring at the start of every item and drains it at the end, so each item pays
// one loaded DRAM round trip with nothing in flight (about 3 us on a GB300
// under full load).  Here one elected thread produces chunk descriptors for
// the items in order -- fetching the next item while the current one is still
// in flight -- and the whole CTA consumes them, so the ring never empties
// between items.  With the shared queue (`a.queue`), CTAs that run faster
// simply take more items, which removes the spread between CTAs that a fixed
// share of bytes leaves (SMs differ in the DRAM bandwidth they get).
//
// Per chunk (Purlin 0.6.5 (PyPI page), "Samples": an Atom copies one aligned
// slice through a pipeline in shared memory):
//   * the producer writes the chunk's descriptor to the slot's entry and
//     issues one bulk load of the chunk's 16-byte-aligned source window,
//     completing on the slot's mbarrier (an item without a 16-byte body gets a
//     descriptor and a bare arrival, so every item passes through the ring);
//   * all threads wait on the mbarrier (which also publishes the descriptor),
//     load the item's head and tail bytes if the chunk is the item's first
//     (stored one chunk later), and, when the source sits m bytes off the
//     destinations' 16-byte grid,
//     cut the destination vectors out of the window with funnel shifts into
//     one of two output tiles;
//   * the producer bulk-stores the chunk (from the slot, or from the tile) to
//     every destination, commits one bulk group, and refills the slot of the
//     previous chunk once that chunk's stores have read it.
// Every wait is bounded; on a time-out the CTA records PL_ERR_TIMEOUT, waits
// (bounded) for the loads it issued and leaves.
#include "kernels_bulk.cuh"

namespace pl {
namespace {

constexpr int kItemRing = 16;           // items referenced by chunks in flight (stages + 2 at most)
constexpr uint32_t kStop = 0xFFFFFFFFu;  // descriptor of the slot after the last chunk

// An item being streamed (shared memory; written by the producer).
struct StreamItem {
  const char* src;          // first source byte
  char* dst[kMaxWorld];     // first byte of each destination
  uint64_t len;             // bytes of the item
  uint64_t head;            // bytes before the destinations' 16-byte boundary
  uint64_t body;            // bytes that go through the ring (a multiple of 16)
  unsigned long long t0;    // trace: when the item was started
  uint32_t nd;              // destinations
  uint32_t index;           // item index (trace)
};

// What a ring slot holds.
struct StreamChunk {
  uint64_t off;             // offset of the chunk in the item's body
  uint32_t item;            // StreamItem entry, or kStop
  uint32_t m;               // body source address mod 16 (0: stores straight from the slot)
  uint32_t len;             // bytes (a multiple of 16; 0 for an item without body)
  uint32_t flags;           // bit 0: the item's first chunk, bit 1: its last
};

__global__ void __launch_bounds__(512, 1) stream_copy_kernel(const __grid_constant__ KArgs a) {
  extern __shared__ __align__(128) char dyn_smem[];
  __shared__ uint64_t full[8];
  __shared__ StreamItem SI[kItemRing];
  __shared__ StreamChunk SC[8];
  grid_dep_wait();

  const uint32_t stages = (uint32_t)a.stages;
  const uint32_t ch = a.chunk_bytes;
  const size_t wslot = (size_t)ch + 16;
  char* const tiles = dyn_smem + (size_t)stages * wslot;
  const bool leader = threadIdx.x == 0;

  // ---- producer state (thread 0 only)
  Item nx{};                // the next item, already loaded
  uint32_t nx_idx = 0;
  bool nx_ok = false;
  uint32_t q_idx = 0;       // queue: index fetched for the item after nx
  uint32_t st_i = 0, st_end = 0;  // static share: items [st_i, st_end)
  uint32_t p_item = 0;      // StreamItem entries used so far
  uint32_t p_cur = 0;       // entry of the item being produced
  const char* p_win = nullptr;
  uint64_t p_off = 0, p_body = 0;
  uint32_t p_m = 0;
  bool p_have = false, p_stopped = false;
  uint32_t issued = 0;      // descriptors published (the stop included)

  // make nx the item after the current one (its load and the next queue
  // fetch complete while the current item streams)
  auto advance = [&]() {
    if (a.queue) {
      nx_ok = q_idx < a.n_items;
      if (nx_ok) {
        nx_idx = q_idx;
        nx = a.items[nx_idx];
        q_idx = gridDim.x + atomicAdd(&a.ctl[kCtlQueue], 1u);
      }
    } else {
      nx_ok = st_i < st_end;
      if (nx_ok) {
        nx_idx = st_i++;
        nx = a.items[nx_idx];
      }
    }
  };

  // publish the next chunk (or the stop) into slot issued % stages
  auto produce = [&]() {
    const uint32_t s = issued % stages;
    if (!p_have) {
      if (!nx_ok) {
        SC[s].item = kStop;
        mbar_expect_tx(&full[s], 0);
        p_stopped = true;
        ++issued;
        return;
      }
      Item it = nx;
      const uint32_t idx = nx_idx;
      advance();
      if (!item_in_bounds(a, it)) {  // checking build: move nothing
        atomicCAS(&a.ctl[kCtlStatus], 0u, (uint32_t)kDevBounds);
        it.len = 0;
      }
      StreamItem& u = SI[p_item % kItemRing];
      p_cur = p_item % kItemRing;
      ++p_item;
      const int b = __ffs(it.src_mask) - 1;
      const char* src = (b < 16 ? a.in[b] : a.out[b - 16]) + it.src_off;
      uint32_t nd = 0;
      for (uint32_t mk = it.dst_mask; mk; mk &= mk - 1) u.dst[nd++] = a.out[__ffs(mk) - 1] + it.dst_off;
      const uint32_t rd = (uint32_t)((uintptr_t)u.dst[0] & 15u);
      const uint64_t head = ((16u - rd) & 15u) < it.len ? ((16u - rd) & 15u) : it.len;
      const uint64_t body = (it.len - head) & ~(uint64_t)15;
      u.src = src;
      u.len = it.len;
      u.head = head;
      u.body = body;
      u.nd = nd;
      u.index = idx;
      u.t0 = a.trace ? globaltimer() : 0ull;
      if (body == 0) {
        // head and tail only: a descriptor and a bare arrival
        SC[s].item = p_cur;
        SC[s].off = 0;
        SC[s].m = 0;
        SC[s].len = 0;
        SC[s].flags = 3u;
        mbar_expect_tx(&full[s], 0);
        ++issued;
        return;
      }
      const char* sb = src + head;
      p_m = (uint32_t)((uintptr_t)sb & 15u);
      p_win = sb - p_m;
      p_off = 0;
      p_body = body;
      p_have = true;
    }
    const uint32_t len = (p_body - p_off) < ch ? (uint32_t)(p_body - p_off) : ch;
    SC[s].item = p_cur;
    SC[s].off = p_off;
    SC[s].m = p_m;
    SC[s].len = len;
    SC[s].flags = (p_off == 0 ? 1u : 0u) | (p_off + len == p_body ? 2u : 0u);
    const uint32_t win = (p_m + len + 15u) & ~15u;
    mbar_expect_tx(&full[s], win);
    bulk_load(dyn_smem + (size_t)s * wslot, p_win + p_off, win, &full[s]);
    p_off += len;
    if (p_off == p_body) p_have = false;
    ++issued;
  };

  if (leader) {
    for (uint32_t i = 0; i < stages; ++i) mbar_init(&full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_shared();
    if (a.queue) {
      q_idx = blockIdx.x;  // CTA c starts with item c; the counter hands out items grid, grid + 1, ...
    } else {
      st_i = a.cta_begin[blockIdx.x];
      st_end = a.cta_begin[blockIdx.x + 1];
    }
    advance();
    for (uint32_t j = 0; j + 1 < stages && !p_stopped; ++j) produce();
  }
  __syncthreads();

  bool failed = false;
  uint32_t shifted = 0;  // shifted chunks so far (tile = shifted % 2); same count in every thread
  // An item's head and tail bytes (fewer than 32, one per thread) are loaded
  // when its first chunk is consumed and stored one chunk later, so the
  // load's L2 latency never holds up the CTA.
  uint32_t hb_item = kStop;
  uint64_t hb_k = 0;
  uint8_t hb_v = 0;
  auto put_byte = [&]() {
    if (hb_item != kStop) {
      const StreamItem& hu = SI[hb_item];
      for (uint32_t j = 0; j < hu.nd; ++j) hu.dst[j][hb_k] = (char)hb_v;
      hb_item = kStop;
    }
  };
  uint32_t c = 0;
  for (;; ++c) {
    const uint32_t s = c % stages;
    const bool ok = mbar_wait(&full[s], (c / stages) & 1u, kBulkWaitNs);
    // one bulk group per chunk: with at most one pending (chunk c-1's), every
    // tile except the one chunk c-1 may have used is free
    if (leader) bulk_wait_read<1>();
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    const StreamChunk q = SC[s];
    if (q.item == kStop) break;
    const StreamItem& u = SI[q.item];
    put_byte();
    if (q.flags & 1u) {
      // the item's head and tail bytes (fewer than 16 each; blockDim.x >= 64)
      const uint64_t tail0 = u.head + u.body;
      const uint32_t nb = (uint32_t)(u.head + (u.len - tail0));
      if (threadIdx.x < nb) {
        hb_k = threadIdx.x < u.head ? threadIdx.x : tail0 + (threadIdx.x - u.head);
        hb_v = ld_byte<true>(u.src + hb_k);
        hb_item = q.item;
      }
    }
    const char* out = dyn_smem + (size_t)s * wslot;
    if (q.m) {
      const uint4* win = reinterpret_cast<const uint4*>(out);
      uint4* tile = reinterpret_cast<uint4*>(tiles + (size_t)(shifted & 1u) * ch);
#pragma unroll 4
      for (uint32_t v = threadIdx.x; v < q.len / 16; v += blockDim.x) tile[v] = window16(win[v], win[v + 1], q.m);
      fence_async_shared();
      out = reinterpret_cast<const char*>(tile);
      ++shifted;
    }
    __syncthreads();
    if (leader) {
      if (q.len)
        for (uint32_t j = 0; j < u.nd; ++j) bulk_store(u.dst[j] + u.head + q.off, out, q.len);
      bulk_commit();  // one group per chunk, empty for an item without body
      if ((q.flags & 2u) && a.trace) trace_put(a, u.t0, globaltimer(), u.index, 0u, u.len);
      // the slot of chunk c-1 is free once its stores have read it
      bulk_wait_read<1>();
      if (!p_stopped) produce();
    }
  }
  put_byte();
  if (leader) {
    if (failed) {
      atomicCAS(&a.ctl[kCtlStatus], 0u, (uint32_t)kDevTimeout);
      // the loads issued after the failing chunk land (or time out) before
      // the shared memory they write goes away
      for (uint32_t j = c + 1; j < issued; ++j) mbar_wait(&full[j % stages], (j / stages) & 1u, kBulkWaitNs);
    }
    bulk_wait_all();
    if (a.queue) {
      // the last CTA to finish resets the queue for the next launch (every
      // CTA has made its last fetch before it counts itself done)
      __threadfence();
      if (atomicAdd(&a.ctl[kCtlQueueDone], 1u) == gridDim.x - 1) {
        a.ctl[kCtlQueue] = 0u;
        a.ctl[kCtlQueueDone] = 0u;
        __threadfence();
      }
    }
  }
}

}  // namespace

const void* kernel_stream_copy() { return (const void*)stream_copy_kernel; }

}  // namespace pl
