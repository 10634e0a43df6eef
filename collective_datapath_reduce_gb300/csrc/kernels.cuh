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

// ------------------------------------------------- item prefetch

// Copy work item `src` (global memory, 8-byte aligned) into shared memory
// `dst` with asynchronous 8-byte copies, so no register holds it while the
// CTA moves the current item.  The issuing thread calls item_prefetch_wait()
// before it reads `dst`.
__device__ __forceinline__ void item_prefetch(Item* dst, const Item* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
#pragma unroll
  for (int k = 0; k < (int)(sizeof(Item) / 8); ++k)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d + 8 * k), "l"(reinterpret_cast<const char*>(src) + 8 * k)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void item_prefetch_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

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
  if (it.dst_mask & kFused) {  // inputs and the reduced destination at src_off, the copy at dst_off
    for (uint32_t m = it.src_mask & 0xFFFFu; m; m &= m - 1)
      if (end > a.in_bytes[__ffs(m) - 1]) return false;
    if (end > a.out_bytes[__ffs(it.dst_mask & kDstRanks) - 1]) return false;
    for (int d = 0; d < a.nsrc; ++d)
      if (it.dst_off + it.len > a.out_bytes[d]) return false;
    return true;
  }
  for (uint32_t m = it.src_mask; m; m &= m - 1) {
    const int b = __ffs(m) - 1;
    if (end > (b < 16 ? a.in_bytes[b] : a.out_bytes[b - 16])) return false;
  }
  for (uint32_t m = it.dst_mask & kDstRanks; m; m &= m - 1)
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

// --------------------------------------------------- ring stages on bf16

// The ring AllReduce over bf16 data keeps its running sum in binary32, as two
// 16-bit halves in two rank outputs (kSplitSrc / kSplitDst items; plan.h).
// A stage adds one bf16 input to that sum (SS: sources are {input, low half,
// high half}) or, at the first stage, adds two inputs (sources {a, b}), and
// stores the new sum as halves (SD: destinations {low, high}) or, at the last
// stage, rounds it once to bf16 (one destination).  The halves were stored
// by another CTA earlier in the launch, so every load goes through the L2.

// Element k of every buffer.
template <bool SS, bool SD>
__device__ __forceinline__ void ring_elem_bf16(const char* const* src, char* const* dst, uint64_t k) {
  const uint64_t o = k * 2;
  float s;
  if (SS) {
    const uint32_t lo = __ldcg(reinterpret_cast<const unsigned short*>(src[1] + o));
    const uint32_t hi = __ldcg(reinterpret_cast<const unsigned short*>(src[2] + o));
    s = __fadd_rn(__uint_as_float((hi << 16) | lo), Elem<bf16_tag>::load_l2(src[0] + o));
  } else {
    s = __fadd_rn(Elem<bf16_tag>::load_l2(src[0] + o), Elem<bf16_tag>::load_l2(src[1] + o));
  }
  if (SD) {
    const uint32_t b = __float_as_uint(s);
    *reinterpret_cast<unsigned short*>(dst[0] + o) = (unsigned short)(b & 0xFFFFu);
    *reinterpret_cast<unsigned short*>(dst[1] + o) = (unsigned short)(b >> 16);
  } else {
    Elem<bf16_tag>::store(dst[0] + o, s);
  }
}

// Two elements held in one 32-bit word of each operand.  x: the bf16 input
// pair (or the first input pair); y / z: the low and high half words of the
// running sums (or, without SS, the second input pair).  Result: the words
// to store, the low and high halves of the new sums (SD), or the pair
// rounded to bf16 in `lo`.
template <bool SS, bool SD>
__device__ __forceinline__ void ring_word(uint32_t x, uint32_t y, uint32_t z, uint32_t& lo, uint32_t& hi) {
  const float x0 = __uint_as_float(x << 16), x1 = __uint_as_float(x & 0xFFFF0000u);
  float s0, s1;
  if (SS) {
    s0 = __fadd_rn(__uint_as_float(__byte_perm(y, z, 0x5410)), x0);
    s1 = __fadd_rn(__uint_as_float(__byte_perm(y, z, 0x7632)), x1);
  } else {
    s0 = __fadd_rn(x0, __uint_as_float(y << 16));
    s1 = __fadd_rn(x1, __uint_as_float(y & 0xFFFF0000u));
  }
  if (SD) {
    lo = __byte_perm(__float_as_uint(s0), __float_as_uint(s1), 0x5410);
    hi = __byte_perm(__float_as_uint(s0), __float_as_uint(s1), 0x7632);
  } else {
    lo = Elem<bf16_tag>::pack2(s0, s1);
    hi = 0u;
  }
}

// One 16-byte vector (8 elements) of every operand: compute and store.
template <bool SS, bool SD, bool STREAMING>
__device__ __forceinline__ void ring_vec_store(uint4 a, uint4 b, uint4 c, uint4* d0, uint4* d1) {
  uint4 lo, hi;
  ring_word<SS, SD>(a.x, b.x, c.x, lo.x, hi.x);
  ring_word<SS, SD>(a.y, b.y, c.y, lo.y, hi.y);
  ring_word<SS, SD>(a.z, b.z, c.z, lo.z, hi.z);
  ring_word<SS, SD>(a.w, b.w, c.w, lo.w, hi.w);
  st_vec<STREAMING>(d0, lo);
  if (SD) st_vec<STREAMING>(d1, hi);
}

// 16-byte vectors [0, nv) at byte offset `off` of every buffer (all buffers
// share one address residue modulo 16); U vectors in flight per thread, all
// loads issued before the first add.
template <bool SS, bool SD, int U, bool STREAMING>
__device__ __forceinline__ void ring_vec_bf16(const char* const* src, char* const* dst, uint64_t off, uint32_t nv) {
  const uint32_t step = blockDim.x;
  const uint4* pa = reinterpret_cast<const uint4*>(src[0] + off);
  const uint4* pb = reinterpret_cast<const uint4*>(src[1] + off);
  const uint4* pc = reinterpret_cast<const uint4*>(src[SS ? 2 : 1] + off);
  uint4* d0 = reinterpret_cast<uint4*>(dst[0] + off);
  uint4* d1 = reinterpret_cast<uint4*>(dst[SD ? 1 : 0] + off);
  uint32_t v = threadIdx.x;
  for (; v + (U - 1) * step < nv; v += U * step) {
    uint4 a[U], b[U], c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      a[u] = ld_l2(pa + v + u * step);
      b[u] = ld_l2(pb + v + u * step);
      c[u] = SS ? ld_l2(pc + v + u * step) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) ring_vec_store<SS, SD, STREAMING>(a[u], b[u], c[u], d0 + v + u * step, d1 + v + u * step);
  }
  for (; v < nv; v += step) {
    const uint4 a = ld_l2(pa + v), b = ld_l2(pb + v);
    const uint4 c = SS ? ld_l2(pc + v) : make_uint4(0u, 0u, 0u, 0u);
    ring_vec_store<SS, SD, STREAMING>(a, b, c, d0 + v, d1 + v);
  }
}

template <bool SS, bool SD, int U, bool STREAMING>
__device__ void ring_stage_bf16(const char* const* src, char* const* dst, uint64_t len) {
  const uint32_t tid = threadIdx.x, nt = blockDim.x;
  const uint64_t n = len / 2;
  const uint32_t res = (uint32_t)((uintptr_t)src[0] & 15u);
  bool co = (((uintptr_t)src[1] & 15u) == res) && (((uintptr_t)dst[0] & 15u) == res);
  if (SS) co = co && (((uintptr_t)src[2] & 15u) == res);
  if (SD) co = co && (((uintptr_t)dst[1] & 15u) == res);
  // buffers at different residues: element by element
  uint64_t head = co ? ((16u - res) & 15u) / 2 : n;
  if (head > n) head = n;
  for (uint64_t k = tid; k < head; k += nt) ring_elem_bf16<SS, SD>(src, dst, k);
  if (head == n) return;
  const uint32_t nv = (uint32_t)(((n - head) * 2) >> 4);
  ring_vec_bf16<SS, SD, U, STREAMING>(src, dst, head * 2, nv);
  for (uint64_t k = head + (uint64_t)nv * 8 + tid; k < n; k += nt) ring_elem_bf16<SS, SD>(src, dst, k);
}

// ------------------------------------------- L2 priorities of SNAC plans

// store_hint 3 (two-shot AllReduce).  A reduce item's inputs are read once:
// loaded with an evict-first L2 policy.  Its result (the owner's tile) is read
// back by the copy items shortly after: stored with an evict-last policy, so
// that the inputs streaming through the L2 do not push it out before the
// copies read it.  The copies load it through the L2, return each line read
// to normal priority, and store their results evict-first (.cs).  Only
// 16-byte aligned items take these paths; any other item runs on the plain
// Atoms.

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 ld_stream_policy(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void st_vec_policy(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

// Return the 128-byte line that starts at p to normal L2 priority; any other
// p (inside a line) does nothing, so that each line is demoted once, by the
// thread that read its first 16 bytes, at the line's own address.
__device__ __forceinline__ void l2_priority_normal(const void* p) {
  if (((uintptr_t)p & 127u) == 0) asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// N-to-1 reduce of a SNAC owner tile with L2 policies (one destination).  NS
// sources known at compile time; falls back to the plain Atom otherwise.
template <typename T, int NS, int U>
__device__ __forceinline__ void reduce_owner_tile(const char* const* src, int ns, char* const* dst, uint64_t len) {
  bool fast = NS > 0 && (len & 15u) == 0 && aligned16(dst[0]);
  for (int s = 0; s < ns; ++s) fast = fast && aligned16(src[s]);
  if constexpr (NS > 0) {
    if (fast) {
      constexpr int EPV = Elem<T>::kPerVec;
      const uint64_t pf = l2_evict_first_policy();
      const uint64_t ps = l2_evict_last_policy();
      const uint32_t nv = (uint32_t)(len >> 4), step = blockDim.x;
      uint32_t v = threadIdx.x;
      auto body = [&](auto uu) {
        constexpr int UU = decltype(uu)::value;
        uint4 r[UU][NS];
#pragma unroll
        for (int b = 0; b < NS; ++b)
#pragma unroll
          for (int u = 0; u < UU; ++u) r[u][b] = ld_stream_policy(reinterpret_cast<const uint4*>(src[b]) + v + u * step, pf);
#pragma unroll
        for (int u = 0; u < UU; ++u) {
          float acc[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) acc[e] = Elem<T>::get(r[u][0], e);
#pragma unroll
          for (int b = 1; b < NS; ++b)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[e] = __fadd_rn(acc[e], Elem<T>::get(r[u][b], e));
          st_vec_policy(reinterpret_cast<uint4*>(dst[0]) + v + u * step, Elem<T>::pack(acc), ps);
        }
      };
      for (; v + (U - 1) * step < nv; v += U * step) body(std::integral_constant<int, U>());
      for (; v < nv; v += step) body(std::integral_constant<int, 1>());
      return;
    }
  }
  reduce_atom<T, NS, U, false, false>(src, ns, dst, 1, len);
}

// Copy of a SNAC owner tile to the other ranks (loads through the L2, each
// line read returned to normal priority, stores evict-first).
__device__ __forceinline__ void copy_owner_tile(const char* src, char* const* dst, int nd, uint64_t len) {
  bool fast = (len & 15u) == 0 && aligned16(src);
  for (int j = 0; j < nd; ++j) fast = fast && aligned16(dst[j]);
  if (!fast) {
    copy_atom<true, 2, true>(src, dst, nd, len);
    return;
  }
  const uint32_t nv = (uint32_t)(len >> 4), step = blockDim.x;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint32_t v = threadIdx.x;
  for (; v + step < nv; v += 2 * step) {
    const uint4 r0 = ld_l2(s4 + v), r1 = ld_l2(s4 + v + step);
    l2_priority_normal(s4 + v);
    l2_priority_normal(s4 + v + step);
    for (int j = 0; j < nd; ++j) {
      uint4* d4 = reinterpret_cast<uint4*>(dst[j]);
      st_vec<true>(d4 + v, r0);
      st_vec<true>(d4 + v + step, r1);
    }
  }
  for (; v < nv; v += step) {
    const uint4 r = ld_l2(s4 + v);
    l2_priority_normal(s4 + v);
    for (int j = 0; j < nd; ++j) st_vec<true>(reinterpret_cast<uint4*>(dst[j]) + v, r);
  }
}

// A fused two-shot item (kFused): reduce the owner tile whose NS sources are
// src[] into dst[0], and in the same pass copy the tile at src_b (another
// CTA's owner tile, reduced earlier in this launch) to dst[1 .. nb]: per
// vector NS + 1 loads and 1 + nb stores, the one-shot layout's mix.  Falls
// back to the two parts one after the other when a pointer is not 16-byte
// aligned or the source count is not known at compile time.
template <typename T, int NS, int U>
__device__ __forceinline__ void fused_owner_tiles(const char* const* src, int ns, char* const* dst, const char* src_b,
                                                  int nb, uint64_t len) {
  if constexpr (NS > 0) {
    bool fast = (len & 15u) == 0 && aligned16(dst[0]) && aligned16(src_b);
    for (int s = 0; s < NS; ++s) fast = fast && aligned16(src[s]);
    for (int j = 1; j <= nb; ++j) fast = fast && aligned16(dst[j]);
    if (fast) {
      constexpr int EPV = Elem<T>::kPerVec;
      const uint64_t pf = l2_evict_first_policy(), pl = l2_evict_last_policy();
      const uint32_t nv = (uint32_t)(len >> 4), step = blockDim.x;
      const uint4* sb = reinterpret_cast<const uint4*>(src_b);
      for (uint32_t v = threadIdx.x; v < nv; v += step) {
        uint4 r[NS];
#pragma unroll
        for (int b = 0; b < NS; ++b) r[b] = ld_stream_policy(reinterpret_cast<const uint4*>(src[b]) + v, pf);
        const uint4 y = ld_l2(sb + v);
        l2_priority_normal(sb + v);
        float acc[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[e] = Elem<T>::get(r[0], e);
#pragma unroll
        for (int b = 1; b < NS; ++b)
#pragma unroll
          for (int e = 0; e < EPV; ++e) acc[e] = __fadd_rn(acc[e], Elem<T>::get(r[b], e));
        st_vec_policy(reinterpret_cast<uint4*>(dst[0]) + v, Elem<T>::pack(acc), pl);
        for (int j = 1; j <= nb; ++j) st_vec<true>(reinterpret_cast<uint4*>(dst[j]) + v, y);
      }
      return;
    }
  }
  reduce_owner_tile<T, NS, U>(src, ns, dst, len);
  copy_owner_tile(src_b, dst + 1, nb, len);
}

// T = void: copy-only kernel (AllGather, AllToAll and their V forms).
// Otherwise items with one source are the consume-side copies of the
// two-shot and ring AllReduce, whose source another CTA produced in this
// launch.  COH: reduce items too may read data produced in this launch (the
// ring's running sums), so their loads go through the L2 rather than the
// non-coherent read-only path.  `split`: the item's kSplitSrc / kSplitDst bits.
template <typename T, int NS, int U, bool STREAMING, bool COH>
__device__ __forceinline__ void run_item(const char* const* src, int ns, char* const* dst, int nd,
                                         uint64_t len, uint32_t split) {
  if constexpr (std::is_same<T, void>::value) {
    copy_atom<false, U, STREAMING>(src[0], dst, nd, len);
  } else {
    if (ns == 1) {
      copy_atom<true, 2, STREAMING>(src[0], dst, nd, len);
    } else if constexpr (COH && std::is_same<T, bf16_tag>::value) {
      if (split == (kSplitSrc | kSplitDst))
        ring_stage_bf16<true, true, U, STREAMING>(src, dst, len);
      else if (split == kSplitSrc)
        ring_stage_bf16<true, false, U, STREAMING>(src, dst, len);
      else if (split == kSplitDst)
        ring_stage_bf16<false, true, U, STREAMING>(src, dst, len);
      else
        reduce_atom<T, NS, U, STREAMING, COH>(src, ns, dst, nd, len);
    } else {
      (void)split;
      reduce_atom<T, NS, U, STREAMING, COH>(src, ns, dst, nd, len);
    }
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

// Kernel kinds.  kKindPlain: every layout but the ring (store_hint 1 or 2).
// kKindRing: the ring's reduce items read running sums stored in this launch.
// kKindL2: SNAC plans with L2 priorities (store_hint 3): owner tiles reduced
// and copied on the paths above.  Each kind is its own instantiation, so the
// others' code never enters the plain kernel.
enum : int { kKindPlain = 0, kKindRing = 1, kKindL2 = 2 };

template <typename T, int NS, int U, int KIND = kKindPlain>
__global__ void __launch_bounds__(snac_max_threads<NS>(), 2) snac_kernel(const __grid_constant__ KArgs a) {
  constexpr bool COH = KIND == kKindRing;
  constexpr uint32_t kNoItem = 0xFFFFFFFFu;
  __shared__ const char* s_src[kMaxWorld];
  __shared__ char* s_dst[kMaxWorld];
  __shared__ uint64_t s_len;
  __shared__ int s_ns, s_nd, s_ok;
  __shared__ uint32_t s_item, s_notify, s_epoch, s_wait_ns, s_split;
  __shared__ const char* s_fsrc;  // fused items: the copied tile
  __shared__ uint32_t s_next_i, s_q_i;  // thread 0's item cursor (kept out of the registers of the Atoms)
  __shared__ __align__(16) Item s_next;  // the next item, prefetched by thread 0
  __shared__ uint32_t s_raised;          // ring: the flag this CTA raised for its last item (0: none)
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
  if constexpr (KIND == kKindRing) {
    if (threadIdx.x == 0) s_raised = 0u;
  }

  // Thread 0 copies the next item into shared memory while the CTA moves the
  // current one (and, on the queue, fetches the index of the item after it).
  if (threadIdx.x == 0) {
    s_next_i = begin;
    s_q_i = 0;
    if (begin < end) {
      item_prefetch(&s_next, a.items + begin);
      if (a.queue) s_q_i = gridDim.x + atomicAdd(&a.ctl[kCtlQueue], 1u);
    }
  }
  for (;;) {
    if (threadIdx.x == 0) {
      s_item = kNoItem;
      const uint32_t i = s_next_i;
      if (i < end) {
        item_prefetch_wait();
        const Item it = s_next;
        const uint32_t ni = a.queue ? s_q_i : i + step;
        s_next_i = ni;
        if (ni < end) {
          item_prefetch(&s_next, a.items + ni);
          if (a.queue) s_q_i = gridDim.x + atomicAdd(&a.ctl[kCtlQueue], 1u);
        }
        s_item = i;
        int ns = 0, nd = 0;
        if (KIND == kKindL2 && (it.dst_mask & kFused)) {
          // reduce the tile at src_off into the one destination bit; copy the
          // tile at dst_off from the output source bit to every other output
          for (uint32_t m = it.src_mask & 0xFFFFu; m; m &= m - 1) s_src[ns++] = a.in[__ffs(m) - 1] + it.src_off;
          const int ob = __ffs(it.src_mask >> 16) - 1;
          s_fsrc = a.out[ob] + it.dst_off;
          s_dst[nd++] = a.out[__ffs(it.dst_mask & kDstRanks) - 1] + it.src_off;
          for (int d = 0; d < a.nsrc; ++d)
            if (d != ob) s_dst[nd++] = a.out[d] + it.dst_off;
        } else {
          for (uint32_t m = it.src_mask; m; m &= m - 1) {
            const int b = __ffs(m) - 1;
            s_src[ns++] = (b < 16 ? a.in[b] : a.out[b - 16]) + it.src_off;
          }
          for (uint32_t m = it.dst_mask & kDstRanks; m; m &= m - 1) s_dst[nd++] = a.out[__ffs(m) - 1] + it.dst_off;
        }
        s_ns = ns;
        s_nd = nd;
        s_split = it.dst_mask & (kSplitSrc | kSplitDst | kFused);
        s_len = it.len;
        if (!item_in_bounds(a, it)) {  // checking build: move nothing, keep the SNAC order
          atomicCAS(&a.ctl[kCtlStatus], 0u, (uint32_t)kDevBounds);
          s_len = 0;
        }
        s_notify = it.notify;
        int ok = 1;
        const unsigned long long t0 = a.trace ? globaltimer() : 0ull;
        if constexpr (KIND == kKindRing) {
          // A tile's stages come one wave apart, so most land on the CTA that
          // ran the stage before: a wait for the flag this CTA raised for
          // its last item is met (its stores are ordered before this item by
          // the block barrier).  Any other wait loads the status word with
          // its first load (one round trip to the L2 for both); a wait that
          // spins reads it again.
          if (it.wait && it.wait != s_raised) {
            const uint32_t status = ld_volatile(&a.ctl[kCtlStatus]);
            ok = consume_wait(a, a.flags + (it.wait - 1), s_epoch);
            if (status != 0) ok = 0;
          }
        } else {
          if (it.wait) ok = consume_wait(a, a.flags + (it.wait - 1), s_epoch);
        }
        s_t0 = t0;
        s_wait_ns = a.trace ? (uint32_t)min(globaltimer() - t0, 0xFFFFFFFFull) : 0u;
        if constexpr (KIND != kKindRing) {
          if (a.sync && ok && ld_volatile(&a.ctl[kCtlStatus]) != 0) ok = 0;
        }
        s_ok = ok;
      }
    }
    __syncthreads();
    const uint32_t i = s_item;
    if (i == kNoItem || !s_ok) break;
    if constexpr (KIND == kKindL2 && !std::is_same<T, void>::value) {
      if (s_split & kFused)
        fused_owner_tiles<T, NS, U>(s_src, s_ns, s_dst, s_fsrc, s_nd - 1, s_len);
      else if (s_ns == 1)
        copy_owner_tile(s_src[0], s_dst, s_nd, s_len);
      else if (s_nd == 1)
        reduce_owner_tile<T, NS, U>(s_src, s_ns, s_dst, s_len);
      else
        run_item<T, NS, U, false, false>(s_src, s_ns, s_dst, s_nd, s_len, s_split);
    } else if (a.store_hint == 2) {
      run_item<T, NS, U, true, COH>(s_src, s_ns, s_dst, s_nd, s_len, s_split);
    } else {
      run_item<T, NS, U, false, COH>(s_src, s_ns, s_dst, s_nd, s_len, s_split);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      if (s_notify && i + 1 != a.drop_notify) {
        // a release is cumulative: it orders every store of the CTA that the
        // barrier ordered before it (the ring's chains of 2 (world - 1)
        // stages per tile go without the extra full fence; the other kinds
        // keep it)
        if constexpr (KIND != kKindRing) __threadfence();
        st_release(a.flags + (s_notify - 1), s_epoch);
      }
      if constexpr (KIND == kKindRing) s_raised = (s_notify && i + 1 != a.drop_notify) ? s_notify : 0u;
      if (a.trace) trace_put(a, s_t0, globaltimer(), i, s_wait_ns, s_len);
    }
  }
  // a loop that stopped at an error may leave the next item's copy in flight
  if (threadIdx.x == 0) item_prefetch_wait();
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
