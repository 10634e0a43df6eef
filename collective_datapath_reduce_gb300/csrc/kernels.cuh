// Device side of the datapath (sm_103a): one persistent kernel per call runs
// the plan's work items with the copy Atom and the N-to-1 reduce Atom, and the
// Stage, Notify And Consume (SNAC) flags between items of one launch.
//
// Purlin README (purlin 0.6.4), "Key Idea": SNAC decides where and when data
// moves, Atoms decide how the GPU moves it.  Here an item names its sources
// and destinations; the Atom chosen by the number of sources moves the bytes:
//   copy Atom   (one source)    dst[j][i] = src[i] for every destination j;
//   reduce Atom (N sources)     dst[j][i] = fold over s of src[s][i], binary32,
//                               ascending source order, starting from source
//                               0's value, one rounding to the output type.
// SNAC (same page, and Iris docs "Device Context", all_reduce_two_shot: ready
// flags between producer and consumer): an item that notifies raises its flag
// to the launch's epoch with a gpu-scope release once every thread of the CTA
// has stored its part; an item that consumes spins with gpu-scope acquire
// loads until its flag holds the epoch, for at most the handle's time limit.
//
// Register path: each thread moves 16-byte vectors, coalesced across the
// warp; all loads of an iteration (U vectors per source) are issued before
// the first add or store, which keeps enough bytes in flight to cover HBM
// latency at 1024 threads per SM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "kargs.h"
#include "purlin_atoms.cuh"

namespace pl {

// --------------------------------------------------------- the SNAC loop

// Spin until *flag == epoch.  Thread 0 only.  Gives up when the time limit
// passes, when the spin count cap is reached, or when another CTA has
// already recorded an error; returns false then.
__device__ __forceinline__ bool consume_wait(const KArgs& a, const uint32_t* flag, uint32_t epoch) {
  const unsigned long long t0 = globaltimer();
  const unsigned long long cap = a.timeout_ns / 16ull + 4096ull;
  for (unsigned long long spin = 0;; ++spin) {
    if (ld_acquire(flag) == epoch) return true;
    if ((spin & 31ull) == 31ull) {
      if (ld_volatile(&a.ctl[kCtlStatus]) != 0) return false;
      if (globaltimer() - t0 > a.timeout_ns || spin > cap) {
        atomicCAS(&a.ctl[kCtlStatus], 0u, (uint32_t)kDevTimeout);
        return false;
      }
    }
    __nanosleep(32);
  }
}

// End of a launch of a plan with SNAC flags; every thread of every CTA calls
// it once its items are done.  The last CTA to get here publishes the
// launch's epoch for the next launch (and resets the shared queue).  Epochs
// run 1, 2, ..., 0xFFFFFFFF and start again at 1: the launch that used
// 0xFFFFFFFF clears every flag of the workspace and publishes 0, so a flag
// written in one cycle can never equal an epoch of the next (flags start at
// 0, and no launch uses epoch 0).
__device__ __forceinline__ void snac_finish(const KArgs& a, uint32_t epoch, bool reset_queue) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&a.ctl[kCtlDone], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  const bool wrap = epoch == 0xFFFFFFFFu;
  if (wrap) {
    for (uint32_t i = threadIdx.x; i < a.flag_cap; i += blockDim.x) a.flags[i] = 0u;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();
    a.ctl[kCtlDone] = 0u;
    a.ctl[kCtlEpoch] = wrap ? 0u : epoch;
    if (reset_queue) a.ctl[kCtlQueue] = 0u;
    __threadfence();
  }
}

// Programmatic dependent launch.  The library launches its kernels with
// programmatic stream serialization, so a launch may start as soon as the
// previous kernel on the stream has retired its CTAs, without waiting for
// the full completion of that grid; grid_dep_wait() returns once that kernel
// has completed and its writes are visible (at once for a plain launch), so
// every kernel calls it before it touches global memory.  No kernel triggers
// its dependents early (griddepcontrol.launch_dependents): measured on a
// GB300 that gained nothing over this.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Checking build (PURLIN_DEBUG): true when every byte item `it` reads and
// writes lies inside the rank buffers' declared sizes.  The normal build
// does not check.
__device__ __forceinline__ bool item_in_bounds(const KArgs& a, const Item& it) {
#ifdef PURLIN_DEBUG
  const uint64_t end = it.src_off + it.len;
  if (end < it.src_off || it.dst_off + it.len < it.dst_off) return false;
  for (uint32_t m = it.src_mask; m; m &= m - 1) {
    const int b = __ffs(m) - 1;
    if (end > (b < 16 ? a.in_bytes[b] : a.out_bytes[b - 16])) return false;
  }
  for (uint32_t m = it.dst_mask; m; m &= m - 1)
    if (it.dst_off + it.len > a.out_bytes[__ffs(m) - 1]) return false;
  return true;
#else
  (void)a;
  (void)it;
  return true;
#endif
}

// Append one record to the trace buffer (thread 0).  Records past the
// capacity are counted but not written.
__device__ __forceinline__ void trace_put(const KArgs& a, unsigned long long t0, unsigned long long t1,
                                          uint32_t item, uint32_t wait_ns, uint64_t len) {
  const unsigned long long slot = atomicAdd(a.trace, 1ull);
  if (slot < a.trace_cap) {
    TraceRecord* r = reinterpret_cast<TraceRecord*>(a.trace + 1) + slot;
    r->t_start = t0;
    r->t_end = t1;
    r->cta = blockIdx.x;
    r->item = item;
    r->wait_ns = wait_ns;
    r->len_kib = (uint32_t)(len >> 10);
  }
}

// T = void: copy-only kernel (AllGather, AllToAll and their V forms).
// Otherwise items with one source are the consume-side copies of the
// two-shot and ring AllReduce, whose source another CTA produced in this
// launch.  COH: reduce items too may read data produced in this launch (the
// ring's partial sums), so their loads go through the L2 rather than the
// non-coherent read-only path.
template <typename T, int NS, int U, bool STREAMING, bool COH>
__device__ __forceinline__ void run_item(const char* const* src, int ns, char* const* dst, int nd,
                                         uint64_t len) {
  if constexpr (std::is_same<T, void>::value) {
    copy_atom<false, U, STREAMING>(src[0], dst, nd, len);
  } else {
    if (ns == 1)
      copy_atom<true, 2, STREAMING>(src[0], dst, nd, len);
    else
      reduce_atom<T, NS, U, STREAMING, COH>(src, ns, dst, nd, len);
  }
}

// Items of a CTA: its contiguous range, every grid-th item (strided SNAC
// plans), or, with the shared queue (`a.queue`), item blockIdx.x first and
// then whatever index the grid-wide counter hands out next.  Every item an
// item waits on comes earlier in the global order, and a CTA only holds (in
// its prefetch registers) an index larger than the one it runs, so the
// earliest unfinished item is always running and the queue cannot deadlock
// a SNAC plan (all CTAs are resident: cooperative launch).
// Launch bound of the register-path kernel: 512 threads for the source
// counts known at compile time; the generic count (up to 16 sources, in
// batches of 8) runs 256-thread CTAs with room for 128 registers, so its 16
// source pointers and 8 vectors in flight stay in registers.
template <int NS>
constexpr int snac_max_threads() { return NS == 0 ? 256 : 512; }

template <typename T, int NS, int U, bool COH = false>
__global__ void __launch_bounds__(snac_max_threads<NS>(), 2) snac_kernel(const __grid_constant__ KArgs a) {
  constexpr uint32_t kNoItem = 0xFFFFFFFFu;
  __shared__ const char* s_src[kMaxWorld];
  __shared__ char* s_dst[kMaxWorld];
  __shared__ uint64_t s_len;
  __shared__ int s_ns, s_nd, s_ok;
  __shared__ uint32_t s_item, s_notify, s_epoch, s_wait_ns;
  __shared__ uint32_t s_next_i, s_q_i;  // thread 0's item cursor (kept out of the registers of the Atoms)
  __shared__ unsigned long long s_t0;
  grid_dep_wait();

  uint32_t begin, end, step;
  if (a.queue) {
    begin = blockIdx.x;
    end = a.n_items;
    step = 0;
  } else if (a.strided) {
    begin = blockIdx.x;
    end = a.n_items;
    step = gridDim.x;
  } else {
    begin = a.cta_begin[blockIdx.x];
    end = a.cta_begin[blockIdx.x + 1];
    step = 1;
  }
  if (threadIdx.x == 0) s_epoch = a.sync ? ld_volatile(&a.ctl[kCtlEpoch]) + 1u : 0u;

  // Thread 0 keeps the next item in registers so its load overlaps the
  // current one (and, on the queue, the index fetched for the item after it).
  Item next;
  if (threadIdx.x == 0) {
    s_next_i = begin;
    s_q_i = 0;
    if (begin < end) {
      next = a.items[begin];
      if (a.queue) s_q_i = gridDim.x + atomicAdd(&a.ctl[kCtlQueue], 1u);
    }
  }
  for (;;) {
    if (threadIdx.x == 0) {
      s_item = kNoItem;
      const uint32_t i = s_next_i;
      if (i < end) {
        const Item it = next;
        const uint32_t ni = a.queue ? s_q_i : i + step;
        s_next_i = ni;
        if (ni < end) {
          next = a.items[ni];
          if (a.queue) s_q_i = gridDim.x + atomicAdd(&a.ctl[kCtlQueue], 1u);
        }
        s_item = i;
        int ns = 0, nd = 0;
        for (uint32_t m = it.src_mask; m; m &= m - 1) {
          const int b = __ffs(m) - 1;
          s_src[ns++] = (b < 16 ? a.in[b] : a.out[b - 16]) + it.src_off;
        }
        for (uint32_t m = it.dst_mask; m; m &= m - 1) s_dst[nd++] = a.out[__ffs(m) - 1] + it.dst_off;
        s_ns = ns;
        s_nd = nd;
        s_len = it.len;
        if (!item_in_bounds(a, it)) {  // checking build: move nothing, keep the SNAC order
          atomicCAS(&a.ctl[kCtlStatus], 0u, (uint32_t)kDevBounds);
          s_len = 0;
        }
        s_notify = it.notify;
        int ok = 1;
        const unsigned long long t0 = a.trace ? globaltimer() : 0ull;
        if (it.wait) ok = consume_wait(a, a.flags + (it.wait - 1), s_epoch);
        s_t0 = t0;
        s_wait_ns = a.trace ? (uint32_t)min(globaltimer() - t0, 0xFFFFFFFFull) : 0u;
        if (a.sync && ok && ld_volatile(&a.ctl[kCtlStatus]) != 0) ok = 0;
        s_ok = ok;
      }
    }
    __syncthreads();
    const uint32_t i = s_item;
    if (i == kNoItem || !s_ok) break;
    if (a.store_hint == 2)
      run_item<T, NS, U, true, COH>(s_src, s_ns, s_dst, s_nd, s_len);
    else
      run_item<T, NS, U, false, COH>(s_src, s_ns, s_dst, s_nd, s_len);
    __syncthreads();
    if (threadIdx.x == 0) {
      if (s_notify && i + 1 != a.drop_notify) {
        __threadfence();
        st_release(a.flags + (s_notify - 1), s_epoch);
      }
      if (a.trace) trace_put(a, s_t0, globaltimer(), i, s_wait_ns, s_len);
    }
  }
  if (a.sync) {
    // (every CTA made its last queue fetch before counting itself done)
    snac_finish(a, s_epoch, a.queue != 0);
  } else if (a.queue) {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(&a.ctl[kCtlQueueDone], 1u) == gridDim.x - 1) {
        a.ctl[kCtlQueue] = 0u;
        a.ctl[kCtlQueueDone] = 0u;
        __threadfence();
      }
    }
  }
}

}  // namespace pl
