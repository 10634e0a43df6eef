// TMA bulk datapath (sm_90+ `cp.async.bulk`, used here on sm_103a): the
// staged alternative to the register path, one work item at a time.  Items
// whose addresses are all 16-byte aligned go through the bulk engines alone;
// copies from a source misaligned against its destinations load aligned
// windows and realign them in shared memory (bulk_copy_shifted_body); other
// misaligned reductions fall back to the register Atoms.  The streamed
// variant for copies (one pipeline across a CTA's items, optional shared
// item queue) is kernels_stream.cu.
//
// Purlin 0.6.5 (PyPI page), "Samples": an Atom copies one aligned slice
// through a pipeline in dynamic shared memory (COPY_PIPELINE_SMEM_BYTES).
// Here that pipeline is a ring of `stages` slots in shared memory:
//   * one elected thread issues 1-D bulk copies global -> shared for every
//     source of a chunk, completing on the slot's mbarrier (transaction bytes);
//   * copy Atom: the same thread then issues one bulk store shared -> global
//     per destination straight from the slot (no register traffic at all);
//   * reduce Atom: all threads wait on the slot's mbarrier, fold the sources
//     from shared memory in ascending order (binary32), round once, write an
//     output tile in shared memory, and the elected thread bulk-stores that
//     tile to every destination.
// Bulk stores are tracked with bulk groups: a slot is refilled only after the
// stores that read it have finished reading (wait_group.read).  Every wait is
// bounded; on time-out the CTA records PL_ERR_TIMEOUT, drains what it issued
// (bounded again) and leaves.
#pragma once

#include "kernels.cuh"

namespace pl {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_read_dyn(int n) {
  switch (n) {
    case 0: bulk_wait_read<0>(); break;
    case 1: bulk_wait_read<1>(); break;
    case 2: bulk_wait_read<2>(); break;
    case 3: bulk_wait_read<3>(); break;
    case 4: bulk_wait_read<4>(); break;
    case 5: bulk_wait_read<5>(); break;
    case 6: bulk_wait_read<6>(); break;
    default: bulk_wait_read<7>(); break;
  }
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Per-CTA pipeline state, kept in shared memory.
struct BulkRing {
  uint64_t full[8];   // one mbarrier per slot
  uint32_t chunk;     // CTA-wide count of chunks started (slot = chunk % stages)
  int failed;         // a wait ran out of time
};

// Pure-TMA copy of the aligned body [0, bytes) of one item: src -> every dst.
// Thread 0 only.  Slots hold `ch` bytes each.
__device__ inline void bulk_copy_body(BulkRing& R, char* ring, int stages, uint32_t ch, const char* src,
                               char* const* dst, int nd, uint64_t bytes, unsigned long long limit_ns) {
  const uint64_t n = (bytes + ch - 1) / ch;
  const uint32_t g0 = R.chunk;
  auto chunk_len = [&](uint64_t k) -> uint32_t {
    const uint64_t off = k * ch;
    return (uint32_t)((bytes - off) < ch ? (bytes - off) : ch);
  };
  auto issue_load = [&](uint64_t k) {
    const uint32_t s = (g0 + (uint32_t)k) % (uint32_t)stages;
    const uint32_t len = chunk_len(k);
    mbar_expect_tx(&R.full[s], len);
    bulk_load(ring + (size_t)s * ch, src + k * ch, len, &R.full[s]);
  };
  const uint64_t pre = n < (uint64_t)(stages - 1) ? n : (uint64_t)(stages - 1);
  for (uint64_t k = 0; k < pre; ++k) issue_load(k);
  uint64_t issued = pre;
  for (uint64_t k = 0; k < n; ++k) {
    const uint32_t g = g0 + (uint32_t)k;
    const uint32_t s = g % (uint32_t)stages;
    if (!mbar_wait(&R.full[s], (g / (uint32_t)stages) & 1u, limit_ns)) {
      R.failed = 1;
      // drain: the loads already issued complete or time out, stores are awaited
      for (uint64_t j = k + 1; j < issued; ++j) {
        const uint32_t gj = g0 + (uint32_t)j;
        mbar_wait(&R.full[gj % (uint32_t)stages], (gj / (uint32_t)stages) & 1u, limit_ns);
      }
      R.chunk = g0 + (uint32_t)issued;
      bulk_wait_read<0>();
      return;
    }
    const uint32_t len = chunk_len(k);
    for (int j = 0; j < nd; ++j) bulk_store(dst[j] + k * ch, ring + (size_t)s * ch, len);
    bulk_commit();
    if (issued < n) {
      // slot of chunk k-1 is refilled once its stores have read it (chunk k's may still be reading)
      bulk_wait_read<1>();
      issue_load(issued);
      ++issued;
    }
  }
  R.chunk = g0 + (uint32_t)n;
}

// Copy whose destinations are 16-byte aligned but whose source sits m bytes
// (1..15) past a 16-byte boundary.  All threads.  Chunk k of the destination
// needs source bytes [k*ch, k*ch + len) = the aligned window starting at
// base + k*ch of round_up(m + len, 16) bytes; the window is loaded with one
// bulk copy (it only spans granules that hold bytes of the source range),
// every thread cuts its destination vectors out of it with funnel shifts into
// an output tile, and the leader bulk-stores the tile.
//
// Shared memory: `stages` windows of ch + 16 bytes, then two output tiles of
// ch bytes used in turn.  A window is refilled as soon as the shift has read
// it, so `stages` loads stay in flight while the stores drain from the tiles;
// tile k % 2 is rewritten only once the stores of chunk k - 2 have read it.
__device__ inline void bulk_copy_shifted_body(BulkRing& R, char* ring, int stages, uint32_t ch, const char* src,
                                       char* const* dst, int nd, uint64_t bytes, unsigned long long limit_ns) {
  const uint32_t m = (uint32_t)((uintptr_t)src & 15u);
  const char* base = src - m;
  const size_t wslot = (size_t)ch + 16;
  char* const otiles = ring + (size_t)stages * wslot;
  const uint64_t n = (bytes + ch - 1) / ch;
  const uint32_t g0 = R.chunk;
  const bool leader = threadIdx.x == 0;
  auto chunk_len = [&](uint64_t k) -> uint32_t {
    const uint64_t off = k * ch;
    return (uint32_t)((bytes - off) < ch ? (bytes - off) : ch);
  };
  auto issue_load = [&](uint64_t k) {
    const uint32_t s = (g0 + (uint32_t)k) % (uint32_t)stages;
    const uint32_t win = (m + chunk_len(k) + 15u) & ~15u;
    mbar_expect_tx(&R.full[s], win);
    bulk_load(ring + s * wslot, base + k * ch, win, &R.full[s]);
  };
  if (leader) {
    const uint64_t pre = n < (uint64_t)stages ? n : (uint64_t)stages;
    for (uint64_t k = 0; k < pre; ++k) issue_load(k);
  }
  uint64_t k = 0;
  for (; k < n; ++k) {
    const uint32_t g = g0 + (uint32_t)k;
    const uint32_t s = g % (uint32_t)stages;
    const bool ok = mbar_wait(&R.full[s], (g / (uint32_t)stages) & 1u, limit_ns);
    // one bulk group per chunk: with at most one pending (chunk k-1), the
    // group of chunk k-2 has read tile k % 2
    if (leader) bulk_wait_read<1>();
    if (__syncthreads_or(!ok)) {
      if (leader) R.failed = 1;
      break;
    }
    const uint32_t len = chunk_len(k);
    const uint4* win = reinterpret_cast<const uint4*>(ring + s * wslot);
    uint4* otile = reinterpret_cast<uint4*>(otiles + (size_t)(k & 1) * ch);
#pragma unroll 4
    for (uint32_t v = threadIdx.x; v < len / 16; v += blockDim.x) otile[v] = window16(win[v], win[v + 1], m);
    fence_async_shared();
    __syncthreads();
    if (leader) {
      for (int j = 0; j < nd; ++j) bulk_store(dst[j] + k * ch, otile, len);
      bulk_commit();
      // every thread has read window s (barrier above): refill it
      if (k + (uint64_t)stages < n) issue_load(k + (uint64_t)stages);
    }
  }
  if (leader) {
    if (R.failed) {
      const uint64_t issued = (k + (uint64_t)stages < n) ? k + (uint64_t)stages : n;
      for (uint64_t j = k + 1; j < issued; ++j) {
        const uint32_t gj = g0 + (uint32_t)j;
        mbar_wait(&R.full[gj % (uint32_t)stages], (gj / (uint32_t)stages) & 1u, limit_ns);
      }
      R.chunk = g0 + (uint32_t)issued;
    } else {
      R.chunk = g0 + (uint32_t)n;
    }
  }
  __syncthreads();
}

// Reduce of the aligned body [0, bytes) of one item.  All threads.
// Slot layout: NSRC input tiles of `ch` bytes, then one output tile.
template <typename T, int NS>
__device__ void bulk_reduce_body(BulkRing& R, char* ring, int stages, uint32_t ch, const char* const* src,
                                 int ns, char* const* dst, int nd, uint64_t bytes, unsigned long long limit_ns) {
  constexpr int EPV = Elem<T>::kPerVec;
  const int nsrc = NS ? NS : ns;
  const size_t slot = (size_t)(nsrc + 1) * ch;
  const uint64_t n = (bytes + ch - 1) / ch;
  const uint32_t g0 = R.chunk;
  const bool leader = threadIdx.x == 0;
  auto chunk_len = [&](uint64_t k) -> uint32_t {
    const uint64_t off = k * ch;
    return (uint32_t)((bytes - off) < ch ? (bytes - off) : ch);
  };
  auto issue_load = [&](uint64_t k) {
    const uint32_t s = (g0 + (uint32_t)k) % (uint32_t)stages;
    const uint32_t len = chunk_len(k);
    char* base = ring + s * slot;
    mbar_expect_tx(&R.full[s], len * (uint32_t)nsrc);
    for (int i = 0; i < nsrc; ++i) bulk_load(base + (size_t)i * ch, src[i] + k * ch, len, &R.full[s]);
  };
  if (leader) {
    const uint64_t pre = n < (uint64_t)stages ? n : (uint64_t)stages;
    for (uint64_t k = 0; k < pre; ++k) issue_load(k);
  }
  uint64_t k = 0;
  for (; k < n; ++k) {
    const uint32_t g = g0 + (uint32_t)k;
    const uint32_t s = g % (uint32_t)stages;
    const bool ok = mbar_wait(&R.full[s], (g / (uint32_t)stages) & 1u, limit_ns);
    if (leader) bulk_wait_read_dyn(stages - 1);  // the output tile of this slot has been read out
    // every thread saw the slot land, or the whole CTA stops
    if (__syncthreads_or(!ok)) {
      if (leader) R.failed = 1;
      break;
    }
    const uint32_t len = chunk_len(k);
    char* base = ring + s * slot;
    char* otile = base + (size_t)nsrc * ch;
    for (uint32_t v = threadIdx.x; v < len / 16; v += blockDim.x) {
      float acc[EPV];
      {
        const uint4 r0 = *reinterpret_cast<const uint4*>(base + (size_t)v * 16);
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[e] = Elem<T>::get(r0, e);
      }
      if (NS) {
#pragma unroll
        for (int i = 1; i < (NS ? NS : 1); ++i) {
          const uint4 r = *reinterpret_cast<const uint4*>(base + (size_t)i * ch + (size_t)v * 16);
#pragma unroll
          for (int e = 0; e < EPV; ++e) acc[e] = __fadd_rn(acc[e], Elem<T>::get(r, e));
        }
      } else {
        for (int i = 1; i < nsrc; ++i) {
          const uint4 r = *reinterpret_cast<const uint4*>(base + (size_t)i * ch + (size_t)v * 16);
#pragma unroll
          for (int e = 0; e < EPV; ++e) acc[e] = __fadd_rn(acc[e], Elem<T>::get(r, e));
        }
      }
      *reinterpret_cast<uint4*>(otile + (size_t)v * 16) = Elem<T>::pack(acc);
    }
    fence_async_shared();
    __syncthreads();
    if (leader) {
      for (int j = 0; j < nd; ++j) bulk_store(dst[j] + k * ch, otile, len);
      bulk_commit();
      if (k + (uint64_t)stages < n) issue_load(k + (uint64_t)stages);
    }
  }
  if (leader) {
    if (R.failed) {
      // drain the loads this item issued beyond the failing chunk
      const uint64_t issued = (k + (uint64_t)stages < n) ? k + (uint64_t)stages : n;
      for (uint64_t j = k + 1; j < issued; ++j) {
        const uint32_t gj = g0 + (uint32_t)j;
        mbar_wait(&R.full[gj % (uint32_t)stages], (gj / (uint32_t)stages) & 1u, limit_ns);
      }
      R.chunk = g0 + (uint32_t)issued;
    } else {
      R.chunk = g0 + (uint32_t)n;
    }
  }
  __syncthreads();
}

// Limit of one mbarrier wait: a bulk copy of a few tens of KiB lands in
// microseconds; one that has not landed after this long never will.
constexpr unsigned long long kBulkWaitNs = 2000000000ull;

template <typename T, int NS>
__global__ void __launch_bounds__(512, 1) bulk_kernel(const __grid_constant__ KArgs a) {
  extern __shared__ __align__(128) char dyn_smem[];
  __shared__ BulkRing R;
  __shared__ const char* s_src[kMaxWorld];
  __shared__ char* s_dst[kMaxWorld];
  __shared__ char* s_dst_body[kMaxWorld];
  __shared__ uint64_t s_len;
  __shared__ int s_ns, s_nd, s_ok, s_aligned;
  __shared__ uint32_t s_notify, s_epoch, s_wait_ns;
  __shared__ unsigned long long s_t0;
  grid_dep_wait();

  const int stages = a.stages;
  const uint32_t ch = a.chunk_bytes;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) mbar_init(&R.full[i], 1);
    R.chunk = 0;
    R.failed = 0;
    s_epoch = a.sync ? ld_volatile(&a.ctl[kCtlEpoch]) + 1u : 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_shared();
  }
  __syncthreads();

  uint32_t begin, end, step;
  if (a.strided) {
    begin = blockIdx.x;
    end = a.n_items;
    step = gridDim.x;
  } else {
    begin = a.cta_begin[blockIdx.x];
    end = a.cta_begin[blockIdx.x + 1];
    step = 1;
  }
  // Thread 0 keeps the next item in registers so its load overlaps the current one.
  Item next;
  if (threadIdx.x == 0 && begin < end) next = a.items[begin];
  for (uint32_t i = begin; i < end; i += step) {
    if (threadIdx.x == 0) {
      const Item it = next;
      if (i + step < end) next = a.items[i + step];
      int ns = 0, nd = 0;
      uintptr_t orr = 0;
      for (uint32_t m = it.src_mask; m; m &= m - 1) {
        const int b = __ffs(m) - 1;
        const char* p = (b < 16 ? a.in[b] : a.out[b - 16]) + it.src_off;
        orr |= (uintptr_t)p;
        s_src[ns++] = p;
      }
      for (uint32_t m = it.dst_mask; m; m &= m - 1) {
        char* p = a.out[__ffs(m) - 1] + it.dst_off;
        orr |= (uintptr_t)p;
        s_dst[nd++] = p;
      }
      s_ns = ns;
      s_nd = nd;
      s_len = it.len;
      if (!item_in_bounds(a, it)) {  // checking build: move nothing, keep the SNAC order
        atomicCAS(&a.ctl[kCtlStatus], 0u, (uint32_t)kDevBounds);
        s_len = 0;
      }
      s_notify = it.notify;
      s_aligned = (orr & 15u) == 0;
      int ok = 1;
      const unsigned long long t0 = a.trace ? globaltimer() : 0ull;
      if (it.wait) {
        ok = consume_wait(a, a.flags + (it.wait - 1), s_epoch);
        fence_async_global();  // the bulk loads below must see what the producer released
      }
      s_t0 = t0;
      s_wait_ns = a.trace ? (uint32_t)min(globaltimer() - t0, 0xFFFFFFFFull) : 0u;
      if (a.sync && ok && ld_volatile(&a.ctl[kCtlStatus]) != 0) ok = 0;
      s_ok = ok && !R.failed;
    }
    __syncthreads();
    if (!s_ok) break;
    const uint64_t len = s_len;
    const int ns = s_ns, nd = s_nd;
    if (!s_aligned && ns == 1) {
      // Copy with misaligned addresses: bytes up to the destinations' 16-byte
      // boundary and the ragged end go through registers, the body through the
      // shifted bulk pipeline.  Loads are L2 loads: the source may be another
      // CTA's output.
      const uint32_t rd = (uint32_t)((uintptr_t)s_dst[0] & 15u);
      const uint64_t head = ((16u - rd) & 15u) < len ? ((16u - rd) & 15u) : len;
      const uint64_t body = (len - head) & ~(uint64_t)15;
      for (uint64_t k = threadIdx.x; k < head; k += blockDim.x) {
        const uint8_t b = ld_byte<true>(s_src[0] + k);
        for (int j = 0; j < nd; ++j) s_dst[j][k] = (char)b;
      }
      for (uint64_t k = head + body + threadIdx.x; k < len; k += blockDim.x) {
        const uint8_t b = ld_byte<true>(s_src[0] + k);
        for (int j = 0; j < nd; ++j) s_dst[j][k] = (char)b;
      }
      if (body) {
        if (threadIdx.x < kMaxWorld) s_dst_body[threadIdx.x] = threadIdx.x < (unsigned)nd ? s_dst[threadIdx.x] + head : nullptr;
        __syncthreads();
        const char* sb = s_src[0] + head;
        if (((uintptr_t)sb & 15u) == 0) {
          if (threadIdx.x == 0) bulk_copy_body(R, dyn_smem, stages, ch, sb, s_dst_body, nd, body, kBulkWaitNs);
        } else {
          bulk_copy_shifted_body(R, dyn_smem, stages, ch, sb, s_dst_body, nd, body, kBulkWaitNs);
        }
      }
    } else if (!s_aligned) {
      // misaligned reductions take the register path
      if constexpr (std::is_same<T, void>::value) {
        copy_atom<false, 4, false>(s_src[0], s_dst, nd, len);
      } else {
        if (ns == 1)
          copy_atom<true, 2, false>(s_src[0], s_dst, nd, len);
        else
          reduce_atom<T, NS, 1, false>(s_src, ns, s_dst, nd, len);
      }
    } else {
      const uint64_t body = len & ~(uint64_t)15;
      if (ns == 1) {
        if (threadIdx.x == 0 && body)
          bulk_copy_body(R, dyn_smem, stages, ch, s_src[0], s_dst, nd, body, kBulkWaitNs);
        // tail bytes (fewer than 16); L2 loads, the source may be another CTA's output
        for (uint64_t k = body + threadIdx.x; k < len; k += blockDim.x) {
          const uint8_t b = ld_byte<true>(s_src[0] + k);
          for (int j = 0; j < nd; ++j) s_dst[j][k] = (char)b;
        }
      } else {
        if constexpr (!std::is_same<T, void>::value) {
          if (body) bulk_reduce_body<T, NS>(R, dyn_smem, stages, ch, s_src, ns, s_dst, nd, body, kBulkWaitNs);
          for (uint64_t k = body / Elem<T>::kBytes + threadIdx.x; k < len / Elem<T>::kBytes; k += blockDim.x)
            reduce_elem<T>(s_src, ns, s_dst, nd, k);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // The next item may lay its slots out differently: let every store of
      // this one finish reading shared memory first.
      bulk_wait_read<0>();
      if (R.failed) atomicCAS(&a.ctl[kCtlStatus], 0u, (uint32_t)kDevTimeout);
      if (s_notify && i + 1 != a.drop_notify) {
        bulk_wait_all();       // this item's bulk stores are complete
        fence_async_global();  // and ordered before the release below
        __threadfence();
        st_release(a.flags + (s_notify - 1), s_epoch);
      }
      if (a.trace) trace_put(a, s_t0, globaltimer(), i, s_wait_ns, s_len);
    }
  }
  if (threadIdx.x == 0) bulk_wait_all();  // shared memory stays valid until every store has read it
  if (a.sync) snac_finish(a, s_epoch, false);
}

}  // namespace pl
