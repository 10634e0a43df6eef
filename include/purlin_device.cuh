// purlin_device.cuh - collectives called from inside a user's kernel.
//
// purlin 0.6.5 (PyPI page), "Device-side": a kernel does some work, fills a
// SnacArgs {bytes, blocks, collBlocks, bIdx} and calls the collective with the
// context created on the host, then does some other work; exactly `blocks`
// CTAs must enter the collective.  This header gives that for the N emulated
// ranks of one GPU: Context holds every rank's source and destination buffer,
// and the collective runs inside the caller's launch:
//
//   1. stage/notify/consume: a grid barrier over the `blocks` CTAs, so that
//      whatever any CTA wrote to the sources before the call is visible;
//   2. the first `coll_blocks` CTAs each take an equal, 512-byte-granular share
//      of the collective's pieces (the same layouts as the host library) and
//      run the copy or N-to-1 reduce Atom on it (purlin_atoms.cuh);
//   3. if `sync_after`, a second barrier, so the caller's work after the call
//      may read any destination.
//
// Every CTA of the launch that enters must enter every collective call, all of
// them must be resident at once (launch cooperatively or keep the grid within
// what fits), and all threads of a CTA call together.  Waits are bounded
// (Context.timeout_ns, 2 s if 0): on time-out the call returns kTimeout
// without moving data, and the two barrier words must be zeroed again before
// they are reused.  Results are bit-identical to the host library's.
#pragma once

#include <type_traits>

#include "purlin_atoms.cuh"

namespace purlin {

constexpr int kMaxRanks = 16;
enum DeviceStatus : int { kOk = 0, kTimeout = 7 };

// The ranks' buffers, filled on the host and passed as a __grid_constant__
// kernel parameter (purlin 0.6.5: `const __grid_constant__ purlin::Context ctx`).
struct Context {
  int world;                      // ranks, 1..16
  const char* src[kMaxRanks];     // rank r's input
  char* dst[kMaxRanks];           // rank r's output
  unsigned int* barrier;          // 2 words of device memory, zero before the first call
  unsigned long long timeout_ns;  // limit of each barrier wait; 0 = 2 s
};

// Per-call arguments (purlin 0.6.5 SnacArgs).  `bytes` follows the host API of
// each collective (per-rank input bytes).
struct SnacArgs {
  unsigned long long bytes;
  int blocks;       // CTAs that enter the call
  int coll_blocks;  // the first coll_blocks of them (by b_idx) move data, 1..blocks
  int b_idx;        // this CTA's index in [0, blocks)
  bool sync_after;  // also barrier after the data are stored
};

namespace detail {

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Generation barrier: word 0 counts arrivals, word 1 is the generation.  The
// last CTA to arrive resets the count and releases the next generation.
__device__ inline int grid_barrier(const Context& c, int blocks) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    ok = 1;
    unsigned* count = c.barrier;
    unsigned* gen = c.barrier + 1;
    __threadfence();
    const unsigned g = *(volatile unsigned*)gen;
    const unsigned arrived = atomicAdd(count, 1u) + 1u;
    if (arrived == (unsigned)blocks) {
      *(volatile unsigned*)count = 0u;
      __threadfence();
      st_release_u32(gen, g + 1u);
    } else {
      const unsigned long long limit = c.timeout_ns ? c.timeout_ns : 2000000000ull;
      const unsigned long long t0 = now_ns();
      for (unsigned spin = 0;; ++spin) {
        if (ld_acquire_u32(gen) != g) break;
        if ((spin & 63u) == 63u && now_ns() - t0 > limit) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
  }
  __syncthreads();
  return ok ? kOk : kTimeout;
}

struct Piece {
  unsigned long long src_off, dst_off, len;
  unsigned src_mask, dst_mask;
};

// This CTA's share of the concatenated pieces (part `part` of `nparts`, cut at
// 512-byte granules of each piece), and the Atom on every overlapped piece.
// `piece(i)` returns piece i; pieces are produced on the fly (no arrays).
template <typename T, int NS, int U, bool STREAMING, class PieceFn>
__device__ void run_share(const Context& c, PieceFn piece, int npieces, int part, int nparts) {
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  unsigned long long W = 0;
  for (int i = 0; i < npieces; ++i) W += piece(i).len;
  auto cut = [&](int j, int& pi, unsigned long long& off) {  // boundary j of nparts
    if (j >= nparts) {
      pi = npieces;
      off = 0;
      return;
    }
    const unsigned long long b = (unsigned long long)(((unsigned __int128)j * W) / (unsigned)nparts);
    unsigned long long start = 0;
    for (pi = 0; pi < npieces && start + piece(pi).len <= b; ++pi) start += piece(pi).len;
    off = pi < npieces ? ((b - start) & ~511ull) : 0;
  };
  int p0, p1;
  unsigned long long o0, o1;
  cut(part, p0, o0);
  cut(part + 1, p1, o1);
  for (int pi = p0; pi <= p1 && pi < npieces; ++pi) {
    const Piece q = piece(pi);
    const unsigned long long a = (pi == p0) ? o0 : 0;
    const unsigned long long e = (pi == p1) ? o1 : q.len;
    if (e <= a) continue;
    __syncthreads();
    if (threadIdx.x == 0) {
      int ns = 0, nd = 0;
      for (unsigned m = q.src_mask; m; m &= m - 1) s_src[ns++] = c.src[__ffs(m) - 1] + q.src_off + a;
      for (unsigned m = q.dst_mask; m; m &= m - 1) s_dst[nd++] = c.dst[__ffs(m) - 1] + q.dst_off + a;
    }
    __syncthreads();
    const int ns = __popc(q.src_mask), nd = __popc(q.dst_mask);
    bool same = true;
    for (int j = 1; j < nd; ++j) same = same && ((((uintptr_t)s_dst[j]) & 15u) == (((uintptr_t)s_dst[0]) & 15u));
    // the sources were written earlier in this launch: coherent (L2) loads
    if (ns == 1) {
      if (same) {
        pl::copy_atom<true, 2, STREAMING>(s_src[0], s_dst, nd, e - a);
      } else {
        for (int j = 0; j < nd; ++j) pl::copy_atom<true, 2, STREAMING>(s_src[0], s_dst + j, 1, e - a);
      }
    } else {
      if constexpr (!std::is_same<T, void>::value) {
        if (same) {
          pl::reduce_atom<T, NS, U, STREAMING, true>(s_src, ns, s_dst, nd, e - a);
        } else {
          for (int j = 0; j < nd; ++j) pl::reduce_atom<T, NS, U, STREAMING, true>(s_src, ns, s_dst + j, 1, e - a);
        }
      }
    }
  }
  __syncthreads();
}

template <typename T, int NS, int U, bool STREAMING, class PieceFn>
__device__ int collective(const SnacArgs& a, const Context& c, PieceFn piece, int npieces) {
  if (grid_barrier(c, a.blocks) != kOk) return kTimeout;
  if (a.b_idx < a.coll_blocks) run_share<T, NS, U, STREAMING>(c, piece, npieces, a.b_idx, a.coll_blocks);
  if (a.sync_after && grid_barrier(c, a.blocks) != kOk) return kTimeout;
  return kOk;
}

__device__ __forceinline__ unsigned all_ranks(int world) { return world >= 32 ? ~0u : ((1u << world) - 1u); }

}  // namespace detail

// AllGather (NKI all_gather_hbm_kernel): dst[r] = src[0] || ... || src[N-1].
// STREAMING (every collective below takes it too): evict-first stores, which
// keep the stored lines from displacing the sources in the L2.
template <bool STREAMING = false>
__device__ inline int all_gather(const SnacArgs& a, const Context& c) {
  const unsigned long long S = a.bytes;
  const unsigned all = detail::all_ranks(c.world);
  auto piece = [=](int s) { return detail::Piece{0ull, s * S, S, 1u << s, all}; };
  return detail::collective<void, 1, 1, STREAMING>(a, c, piece, c.world);
}

// AllToAll (NKI all_to_all_hbm_kernel): chunk d of src[s] -> chunk s of dst[d];
// bytes must split into world chunks.
template <bool STREAMING = false>
__device__ inline int all_to_all(const SnacArgs& a, const Context& c) {
  const int N = c.world;
  const unsigned long long ch = a.bytes / (unsigned)N;
  auto piece = [=](int i) {
    const int s = i / N, d = i % N;
    return detail::Piece{d * ch, s * ch, ch, 1u << s, 1u << d};
  };
  return detail::collective<void, 1, 1, STREAMING>(a, c, piece, N * N);
}

// AllReduce (NKI all_reduce_hbm_kernel), one-shot layout: T = float or
// pl::bf16_tag; NS = world if known at compile time (2..8), else 0; U =
// 16-byte vectors each thread keeps in flight per source.
template <typename T, int NS = 0, int U = 2, bool STREAMING = false>
__device__ int all_reduce(const SnacArgs& a, const Context& c) {
  const unsigned all = detail::all_ranks(c.world);
  const unsigned long long S = a.bytes;
  auto piece = [=](int) { return detail::Piece{0ull, 0ull, S, all, all}; };
  return detail::collective<T, NS, U, STREAMING>(a, c, piece, 1);
}

// ReduceScatter (NKI reduce_scatter_hbm_kernel): dst[r] = chunk r of the sum;
// bytes (per-rank input) must split into world chunks of whole elements.
template <typename T, int NS = 0, int U = 2, bool STREAMING = false>
__device__ int reduce_scatter(const SnacArgs& a, const Context& c) {
  const unsigned long long ch = a.bytes / (unsigned)c.world;
  const unsigned all = detail::all_ranks(c.world);
  auto piece = [=](int r) { return detail::Piece{r * ch, 0ull, ch, all, 1u << r}; };
  return detail::collective<T, NS, U, STREAMING>(a, c, piece, c.world);
}

}  // namespace purlin
