// purlin_atoms.cuh - the datapath Atoms for sm_103a, as device functions.
//
// Purlin README (purlin 0.6.4): underneath the collectives are two
// hardware-aware primitives, a copy and an N-to-1 reduce that combines several
// input buffers into one output; purlin 0.6.5 (PyPI page), "Device-side" and
// "Samples": the threads of a CTA call an Atom on one slice, from any kernel.
// These are those two Atoms (register path) for CUDA C++ code compiled with
// nvcc for sm_103a; the library's own kernels are built from them too.
//
//   pl::copy_atom<COHERENT, U, STREAMING>(src, dst[], nd, len)
//       dst[j][0..len) = src[0..len) for j < nd; any byte alignment; every
//       dst[j] must have the same address modulo 16.  COHERENT: the source was
//       written by another CTA of the same launch (loads go to L2).
//   pl::reduce_atom<T, NS, U, STREAMING>(src[], ns, dst[], nd, len)
//       dst[j][i] = fold over s < ns of src[s][i]: binary32 adds in ascending
//       source order from src[0]'s value, one rounding to T (float or
//       pl::bf16_tag); pointers aligned to the element size, every dst[j] with
//       the same address modulo 16.  NS = ns when the
//       count is known at compile time (2..8), else 0.  A fifth template
//       argument COHERENT = true makes the loads L2 loads, for sources written
//       earlier in the same launch.
//
// Both are called by every thread of the CTA (threadIdx.x / blockDim.x split
// the work) and return when this CTA's stores are issued.  `src` / `dst`
// arrays may live in shared memory.  U: 16-byte vectors in flight per thread
// per source.  STREAMING: evict-first stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

// A 16-byte vector stored as pieces of SW bytes (16, 8, 4 or 2): for
// destinations aligned only to SW.
template <bool STREAMING, int SW>
__device__ __forceinline__ void st_parts(void* p, uint4 v) {
  if constexpr (SW == 16) {
    st_vec<STREAMING>(p, v);
  } else if constexpr (SW == 8) {
    if (STREAMING) {
      asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
      asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"((char*)p + 8), "r"(v.z), "r"(v.w) : "memory");
    } else {
      asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
      asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"((char*)p + 8), "r"(v.z), "r"(v.w) : "memory");
    }
  } else if constexpr (SW == 4) {
    uint32_t* q = reinterpret_cast<uint32_t*>(p);
    q[0] = v.x;
    q[1] = v.y;
    q[2] = v.z;
    q[3] = v.w;
  } else {
    unsigned short* q = reinterpret_cast<unsigned short*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      q[2 * i] = (unsigned short)(w[i] & 0xFFFFu);
      q[2 * i + 1] = (unsigned short)(w[i] >> 16);
    }
  }
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
  __device__ static float load_l2(const char* p) { return __ldcg(reinterpret_cast<const float*>(p)); }
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
  __device__ static float load_l2(const char* p) {
    return __bfloat162float(__ushort_as_bfloat16(__ldcg(reinterpret_cast<const unsigned short*>(p))));
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
template <typename T, bool COHERENT = false>
__device__ __forceinline__ void reduce_elem(const char* const* src, int ns, char* const* dst, int nd,
                                            uint64_t k) {
  const uint64_t o = k * Elem<T>::kBytes;
  float acc = COHERENT ? Elem<T>::load_l2(src[0] + o) : Elem<T>::load(src[0] + o);
  for (int s = 1; s < ns; ++s)
    acc = __fadd_rn(acc, COHERENT ? Elem<T>::load_l2(src[s] + o) : Elem<T>::load(src[s] + o));
  for (int j = 0; j < nd; ++j) Elem<T>::store(dst[j] + o, acc);
}

// Fold K sources (vectors v, v + step, ... of each) into acc: all K x UU
// loads first, then the adds in source order.  FIRST: acc starts from the
// first source's values.
template <typename T, int K, int UU, bool FIRST, bool COHERENT>
__device__ __forceinline__ void fold_batch(const char* const* src, uint64_t off, uint32_t v, uint32_t step,
                                           float (&acc)[UU][Elem<T>::kPerVec]) {
  constexpr int EPV = Elem<T>::kPerVec;
  uint4 r[UU][K];
#pragma unroll
  for (int b = 0; b < K; ++b) {
    const uint4* p = reinterpret_cast<const uint4*>(src[b] + off) + v;
#pragma unroll
    for (int u = 0; u < UU; ++u) r[u][b] = ld_vec<COHERENT>(p + u * step);
  }
#pragma unroll
  for (int u = 0; u < UU; ++u) {
#pragma unroll
    for (int b = 0; b < K; ++b) {
      if (FIRST && b == 0) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[u][e] = Elem<T>::get(r[u][b], e);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[u][e] = __fadd_rn(acc[u][e], Elem<T>::get(r[u][b], e));
      }
    }
  }
}

// Fold a run-time count of 1..8 sources, each count with its own unrolled code.
template <typename T, int UU, bool FIRST, bool COHERENT>
__device__ __forceinline__ void fold_up_to_8(const char* const* src, int k, uint64_t off, uint32_t v,
                                             uint32_t step, float (&acc)[UU][Elem<T>::kPerVec]) {
  switch (k) {
    case 1: fold_batch<T, 1, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
    case 2: fold_batch<T, 2, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
    case 3: fold_batch<T, 3, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
    case 4: fold_batch<T, 4, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
    case 5: fold_batch<T, 5, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
    case 6: fold_batch<T, 6, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
    case 7: fold_batch<T, 7, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
    default: fold_batch<T, 8, UU, FIRST, COHERENT>(src, off, v, step, acc); break;
  }
}

// UU vectors starting at index v (stride `step`) of every source: fold and
// store.  NS > 0: exactly NS sources, all loads issued before the first add.
// NS == 0: ns sources (1..16): the first up to 8 as one batch, the rest as a
// second, each batch with all its loads issued before its adds.
template <typename T, int NS, int UU, bool STREAMING, bool COHERENT = false, int SW = 16>
__device__ __forceinline__ void reduce_step(const char* const* src, int ns, char* const* dst, int nd,
                                            uint64_t off, uint32_t v, uint32_t step) {
  constexpr int EPV = Elem<T>::kPerVec;
  float acc[UU][EPV];
  if constexpr (NS > 0) {
    fold_batch<T, NS, UU, true, COHERENT>(src, off, v, step, acc);
  } else {
    fold_up_to_8<T, UU, true, COHERENT>(src, ns < 8 ? ns : 8, off, v, step, acc);
    if (ns > 8) fold_up_to_8<T, UU, false, COHERENT>(src + 8, ns - 8, off, v, step, acc);
  }
#pragma unroll
  for (int u = 0; u < UU; ++u) {
    const uint4 o = Elem<T>::pack(acc[u]);
    for (int j = 0; j < nd; ++j) st_parts<STREAMING, SW>(dst[j] + off + (uint64_t)(v + u * step) * 16, o);
  }
}

template <typename T, int NS, int U, bool STREAMING, bool COHERENT = false, int SW = 16>
__device__ __forceinline__ void reduce_vec(const char* const* src, int ns, char* const* dst, int nd,
                                           uint64_t off, uint32_t nv) {
  const uint32_t step = blockDim.x;
  uint32_t v = threadIdx.x;
  for (; v + (U - 1) * step < nv; v += U * step)
    reduce_step<T, NS, U, STREAMING, COHERENT, SW>(src, ns, dst, nd, off, v, step);
  if (U > 1)
    for (; v < nv; v += step) reduce_step<T, NS, 1, STREAMING, COHERENT, SW>(src, ns, dst, nd, off, v, step);
}

template <typename T, int NS, int U, bool STREAMING, bool COHERENT = false>
__device__ void reduce_atom(const char* const* src, int ns, char* const* dst, int nd, uint64_t len) {
  constexpr uint64_t E = Elem<T>::kBytes;
  const uint32_t tid = threadIdx.x, nt = blockDim.x;
  const uint64_t n = len / E;
  const uint32_t res = (uint32_t)((uintptr_t)src[0] & 15u);
  bool co = true;
  for (int s = 1; s < ns; ++s) co = co && (((uintptr_t)src[s] & 15u) == res);
  if (!co) {
    for (uint64_t k = tid; k < n; k += nt) reduce_elem<T, COHERENT>(src, ns, dst, nd, k);
    return;
  }
  // Vectors follow the sources' 16-byte alignment; the destinations (one
  // residue for all of them) get each vector in the widest stores their
  // alignment allows.
  uint64_t head = ((16u - res) & 15u) / E;
  if (head > n) head = n;
  for (uint64_t k = tid; k < head; k += nt) reduce_elem<T, COHERENT>(src, ns, dst, nd, k);
  const uint32_t nv = (uint32_t)(((n - head) * E) >> 4);
  const uint32_t rd = (uint32_t)(((uintptr_t)dst[0] + head * E) & 15u);
  if (rd == 0)
    reduce_vec<T, NS, U, STREAMING, COHERENT, 16>(src, ns, dst, nd, head * E, nv);
  else if ((rd & 7u) == 0)
    reduce_vec<T, NS, U, STREAMING, COHERENT, 8>(src, ns, dst, nd, head * E, nv);
  else if ((rd & 3u) == 0)
    reduce_vec<T, NS, U, STREAMING, COHERENT, 4>(src, ns, dst, nd, head * E, nv);
  else
    reduce_vec<T, NS, U, STREAMING, COHERENT, 2>(src, ns, dst, nd, head * E, nv);
  for (uint64_t k = head + (uint64_t)nv * (16 / E) + tid; k < n; k += nt)
    reduce_elem<T, COHERENT>(src, ns, dst, nd, k);
}

}  // namespace pl
