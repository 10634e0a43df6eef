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

namespace pl {

// ------------------------------------------------------------ memory ops

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Loads of data another CTA of the same launch produced: served by L2.
__device__ __forceinline__ uint4 ld_l2(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool COHERENT>
__device__ __forceinline__ uint4 ld_vec(const void* p) {
  if (COHERENT) return ld_l2(p);
  return ld_stream(p);
}

// Shifted copies read every granule twice (two neighbouring threads), so
// these loads may allocate in L1.
template <bool COHERENT>
__device__ __forceinline__ uint4 ld_vec_shared(const uint4* p) {
  if (COHERENT) return ld_l2(p);
  return __ldg(p);
}

template <bool COHERENT>
__device__ __forceinline__ uint8_t ld_byte(const char* p) {
  if (COHERENT) return (uint8_t)__ldcg((const unsigned char*)p);
  return (uint8_t)__ldg((const unsigned char*)p);
}

template <bool STREAMING>
__device__ __forceinline__ void st_vec(void* p, uint4 v) {
  if (STREAMING)
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
  else
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile(const uint32_t* p) {
  return *(const volatile uint32_t*)p;
}

// The 16 bytes that start m bytes into the 32-byte window A:B (m in 1..15).
__device__ __forceinline__ uint4 window16(uint4 A, uint4 B, uint32_t m) {
  const uint32_t sh = (m & 3u) * 8u;
  uint32_t w0, w1, w2, w3, w4;
  switch (m >> 2) {
    case 0: w0 = A.x; w1 = A.y; w2 = A.z; w3 = A.w; w4 = B.x; break;
    case 1: w0 = A.y; w1 = A.z; w2 = A.w; w3 = B.x; w4 = B.y; break;
    case 2: w0 = A.z; w1 = A.w; w2 = B.x; w3 = B.y; w4 = B.z; break;
    default: w0 = A.w; w1 = B.x; w2 = B.y; w3 = B.z; w4 = B.w; break;
  }
  uint4 o;
  o.x = __funnelshift_r(w0, w1, sh);
  o.y = __funnelshift_r(w1, w2, sh);
  o.z = __funnelshift_r(w2, w3, sh);
  o.w = __funnelshift_r(w3, w4, sh);
  return o;
}

// ------------------------------------------------------------- copy Atom

// Vector body of a copy whose source and destinations are 16-byte aligned:
// vectors [0, nv) of s4 to vectors [0, nv) of every dst[j] + off.
template <bool COHERENT, int U, bool STREAMING>
__device__ __forceinline__ void copy_vec(const uint4* s4, char* const* dst, int nd, uint64_t off,
                                         uint32_t nv) {
  const uint32_t step = blockDim.x;
  uint32_t v = threadIdx.x;
  for (; v + (U - 1) * step < nv; v += U * step) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = ld_vec<COHERENT>(s4 + v + u * step);
    for (int j = 0; j < nd; ++j) {
      uint4* d4 = reinterpret_cast<uint4*>(dst[j] + off) + v;
#pragma unroll
      for (int u = 0; u < U; ++u) st_vec<STREAMING>(d4 + u * step, r[u]);
    }
  }
  for (; v < nv; v += step) {
    const uint4 r = ld_vec<COHERENT>(s4 + v);
    for (int j = 0; j < nd; ++j) st_vec<STREAMING>(reinterpret_cast<uint4*>(dst[j] + off) + v, r);
  }
}

// Vector body of a copy whose destinations are aligned and whose source sits
// m bytes past a 16-byte boundary: each destination vector is cut from the
// two aligned source granules that hold its bytes.  Both granules hold bytes
// of the source range, so no load touches a granule outside the buffer.
template <bool COHERENT, bool STREAMING>
__device__ __forceinline__ void copy_vec_shifted(const uint4* sa, uint32_t m, char* const* dst, int nd,
                                                 uint64_t off, uint32_t nv) {
  const uint32_t step = blockDim.x;
  for (uint32_t v = threadIdx.x; v < nv; v += step) {
    const uint4 A = ld_vec_shared<COHERENT>(sa + v);
    const uint4 B = ld_vec_shared<COHERENT>(sa + v + 1);
    const uint4 r = window16(A, B, m);
    for (int j = 0; j < nd; ++j) st_vec<STREAMING>(reinterpret_cast<uint4*>(dst[j] + off) + v, r);
  }
}

// dst[j][0..len) = src[0..len) for j < nd.  All destinations share one
// address residue modulo 16 (the layout engine groups them that way).
template <bool COHERENT, int U, bool STREAMING>
__device__ void copy_atom(const char* src, char* const* dst, int nd, uint64_t len) {
  const uint32_t tid = threadIdx.x, nt = blockDim.x;
  const uint32_t rd = (uint32_t)((uintptr_t)dst[0] & 15u);
  uint32_t head = (16u - rd) & 15u;
  if (head > len) head = (uint32_t)len;
  for (uint32_t k = tid; k < head; k += nt) {
    const uint8_t b = ld_byte<COHERENT>(src + k);
    for (int j = 0; j < nd; ++j) dst[j][k] = (char)b;
  }
  const uint32_t nv = (uint32_t)((len - head) >> 4);
  const char* s = src + head;
  const uint32_t m = (uint32_t)((uintptr_t)s & 15u);
  if (m == 0)
    copy_vec<COHERENT, U, STREAMING>(reinterpret_cast<const uint4*>(s), dst, nd, head, nv);
  else
    copy_vec_shifted<COHERENT, STREAMING>(reinterpret_cast<const uint4*>(s - m), m, dst, nd, head, nv);
  for (uint64_t k = head + ((uint64_t)nv << 4) + tid; k < len; k += nt) {
    const uint8_t b = ld_byte<COHERENT>(src + k);
    for (int j = 0; j < nd; ++j) dst[j][k] = (char)b;
  }
}

// ----------------------------------------------------------- reduce Atom

struct bf16_tag {};

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  static constexpr int kPerVec = 4;
  __device__ static float load(const char* p) { return __ldg(reinterpret_cast<const float*>(p)); }
  __device__ static void store(char* p, float v) { *reinterpret_cast<float*>(p) = v; }
  __device__ static float get(const uint4& r, int e) {
    const uint32_t w = e == 0 ? r.x : e == 1 ? r.y : e == 2 ? r.z : r.w;
    return __uint_as_float(w);
  }
  __device__ static uint4 pack(const float* a) {
    return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                      __float_as_uint(a[3]));
  }
};

template <>
struct Elem<bf16_tag> {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;
  __device__ static float load(const char* p) {
    return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p)));
  }
  __device__ static void store(char* p, float v) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
  }
  // element e of the 8 packed in r (little-endian: element 2k is the low half of word k)
  __device__ static float get(const uint4& r, int e) {
    const uint32_t w = (e >> 1) == 0 ? r.x : (e >> 1) == 1 ? r.y : (e >> 1) == 2 ? r.z : r.w;
    const unsigned short h = (e & 1) ? (unsigned short)(w >> 16) : (unsigned short)(w & 0xFFFFu);
    return __bfloat162float(__ushort_as_bfloat16(h));
  }
  __device__ static uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static uint4 pack(const float* a) {
    return make_uint4(pack2(a[0], a[1]), pack2(a[2], a[3]), pack2(a[4], a[5]), pack2(a[6], a[7]));
  }
};

// Element-by-element fold for heads, tails and sources that are not
// co-aligned.  Element k of every buffer.
template <typename T>
__device__ __forceinline__ void reduce_elem(const char* const* src, int ns, char* const* dst, int nd,
                                            uint64_t k) {
  const uint64_t o = k * Elem<T>::kBytes;
  float acc = Elem<T>::load(src[0] + o);
  for (int s = 1; s < ns; ++s) acc = __fadd_rn(acc, Elem<T>::load(src[s] + o));
  for (int j = 0; j < nd; ++j) Elem<T>::store(dst[j] + o, acc);
}

// UU vectors starting at index v (stride `step`) of every source: fold and
// store.  NS > 0: exactly NS sources, all loads issued before the first add.
// NS == 0: ns sources (up to 16), loaded in batches of 8.
template <typename T, int NS, int UU, bool STREAMING>
__device__ __forceinline__ void reduce_step(const char* const* src, int ns, char* const* dst, int nd,
                                            uint64_t off, uint32_t v, uint32_t step) {
  constexpr int EPV = Elem<T>::kPerVec;
  constexpr int B = NS ? NS : 8;
  const int nsrc = NS ? NS : ns;
  float acc[UU][EPV];
  for (int s0 = 0; s0 < nsrc; s0 += B) {
    uint4 r[UU][B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (NS || s0 + b < nsrc) {
        const uint4* p = reinterpret_cast<const uint4*>(src[s0 + b] + off) + v;
#pragma unroll
        for (int u = 0; u < UU; ++u) r[u][b] = ld_stream(p + u * step);
      }
    }
#pragma unroll
    for (int u = 0; u < UU; ++u) {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (NS || s0 + b < nsrc) {
          if (s0 + b == 0) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[u][e] = Elem<T>::get(r[u][b], e);
          } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[u][e] = __fadd_rn(acc[u][e], Elem<T>::get(r[u][b], e));
          }
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < UU; ++u) {
    const uint4 o = Elem<T>::pack(acc[u]);
    for (int j = 0; j < nd; ++j)
      st_vec<STREAMING>(reinterpret_cast<uint4*>(dst[j] + off) + v + u * step, o);
  }
}

template <typename T, int NS, int U, bool STREAMING>
__device__ __forceinline__ void reduce_vec(const char* const* src, int ns, char* const* dst, int nd,
                                           uint64_t off, uint32_t nv) {
  const uint32_t step = blockDim.x;
  uint32_t v = threadIdx.x;
  for (; v + (U - 1) * step < nv; v += U * step) reduce_step<T, NS, U, STREAMING>(src, ns, dst, nd, off, v, step);
  if (U > 1)
    for (; v < nv; v += step) reduce_step<T, NS, 1, STREAMING>(src, ns, dst, nd, off, v, step);
}

template <typename T, int NS, int U, bool STREAMING>
__device__ void reduce_atom(const char* const* src, int ns, char* const* dst, int nd, uint64_t len) {
  constexpr uint64_t E = Elem<T>::kBytes;
  const uint32_t tid = threadIdx.x, nt = blockDim.x;
  const uint64_t n = len / E;
  const uint32_t res = (uint32_t)((uintptr_t)src[0] & 15u);
  bool co = ((uintptr_t)dst[0] & 15u) == res;
  for (int s = 1; s < ns; ++s) co = co && (((uintptr_t)src[s] & 15u) == res);
  if (!co) {
    for (uint64_t k = tid; k < n; k += nt) reduce_elem<T>(src, ns, dst, nd, k);
    return;
  }
  uint64_t head = ((16u - res) & 15u) / E;
  if (head > n) head = n;
  for (uint64_t k = tid; k < head; k += nt) reduce_elem<T>(src, ns, dst, nd, k);
  const uint32_t nv = (uint32_t)(((n - head) * E) >> 4);
  reduce_vec<T, NS, U, STREAMING>(src, ns, dst, nd, head * E, nv);
  for (uint64_t k = head + (uint64_t)nv * (16 / E) + tid; k < n; k += nt)
    reduce_elem<T>(src, ns, dst, nd, k);
}

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
// two-shot AllReduce, whose source another CTA produced in this launch.
template <typename T, int NS, int U, bool STREAMING>
__device__ __forceinline__ void run_item(const char* const* src, int ns, char* const* dst, int nd,
                                         uint64_t len) {
  if constexpr (std::is_same<T, void>::value) {
    copy_atom<false, U, STREAMING>(src[0], dst, nd, len);
  } else {
    if (ns == 1)
      copy_atom<true, 2, STREAMING>(src[0], dst, nd, len);
    else
      reduce_atom<T, NS, U, STREAMING>(src, ns, dst, nd, len);
  }
}

template <typename T, int NS, int U>
__global__ void __launch_bounds__(512, 2) snac_kernel(const __grid_constant__ KArgs a) {
  __shared__ const char* s_src[kMaxWorld];
  __shared__ char* s_dst[kMaxWorld];
  __shared__ uint64_t s_len;
  __shared__ int s_ns, s_nd, s_ok;
  __shared__ uint32_t s_notify, s_epoch, s_wait_ns;
  __shared__ unsigned long long s_t0;

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
  if (threadIdx.x == 0) s_epoch = a.sync ? ld_volatile(&a.ctl[kCtlEpoch]) + 1u : 0u;

  // Thread 0 keeps the next item in registers so its load overlaps the current one.
  Item next;
  if (threadIdx.x == 0 && begin < end) next = a.items[begin];
  for (uint32_t i = begin; i < end; i += step) {
    if (threadIdx.x == 0) {
      const Item it = next;
      if (i + step < end) next = a.items[i + step];
      int ns = 0, nd = 0;
      for (uint32_t m = it.src_mask; m; m &= m - 1) {
        const int b = __ffs(m) - 1;
        s_src[ns++] = (b < 16 ? a.in[b] : a.out[b - 16]) + it.src_off;
      }
      for (uint32_t m = it.dst_mask; m; m &= m - 1) s_dst[nd++] = a.out[__ffs(m) - 1] + it.dst_off;
      s_ns = ns;
      s_nd = nd;
      s_len = it.len;
      s_notify = it.notify;
      int ok = 1;
      const unsigned long long t0 = a.trace ? globaltimer() : 0ull;
      if (it.wait) ok = consume_wait(a, a.flags + (it.wait - 1), s_epoch);
      s_t0 = t0;
      s_wait_ns = a.trace ? (uint32_t)min(globaltimer() - t0, 0xFFFFFFFFull) : 0u;
      if (a.sync && ok && ld_volatile(&a.ctl[kCtlStatus]) != 0) ok = 0;
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) break;
    if (a.store_hint == 2)
      run_item<T, NS, U, true>(s_src, s_ns, s_dst, s_nd, s_len);
    else
      run_item<T, NS, U, false>(s_src, s_ns, s_dst, s_nd, s_len);
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
    // The last CTA to finish publishes the launch's epoch for the next one.
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const uint32_t done = atomicAdd(&a.ctl[kCtlDone], 1u);
      if (done == gridDim.x - 1) {
        a.ctl[kCtlDone] = 0u;
        a.ctl[kCtlEpoch] = s_epoch;
        __threadfence();
      }
    }
  }
}

}  // namespace pl
