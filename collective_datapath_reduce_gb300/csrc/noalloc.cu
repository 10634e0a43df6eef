// AllReduce that allocates nothing: purlin_all_reduce_noalloc.
//
// Some callers may not allocate device memory once they are running: a
// runtime that fixes its memory at start-up, a plug-in that lives inside
// another framework's memory pool and must not go around it, or code that
// cannot afford the device-wide synchronisation cudaMalloc / cudaFree may
// imply.  They cannot create a handle (its workspace and cached plans are
// allocated).  This entry point runs the two-shot AllReduce without a handle:
// its scratch (SNAC flags and control words) is the file-scope array below,
// and the work items are computed in the kernel instead of being uploaded.
//
// The array lives in every GPU that loads the library until the process
// exits.  Every call on a device shares it and it keeps the last call's
// contents; flags carry the launch's epoch, so stale values never match and
// nothing has to be cleared between calls (except once every 2^32 - 1 calls,
// when the epoch wraps and the last launch of the cycle clears the flags).  Calls that overlap on the GPU
// (different streams, no ordering) race on the array and must not be made.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "kernels.cuh"
#include "purlin_gb.h"

namespace pl {
namespace {

// Control words, then one flag per two-shot tile.
constexpr int kNaCtlWords = 64;
constexpr int kNaMaxFlags = 16384;
constexpr uint64_t kNaTile = 64 * 1024;  // bytes of one owner's range per tile
constexpr int kNaMaxDevices = 64;
constexpr int kNaThreads = 512;
enum : int { kNaEpoch = 0, kNaFailed = 1, kNaDone = 2 };

static __device__ __align__(256) uint32_t g_noalloc_scratch[kNaCtlWords + kNaMaxFlags];

struct NaArgs {
  const char* in[kMaxWorld];
  char* out[kMaxWorld];
  uint32_t* scratch;         // device address of g_noalloc_scratch
  int* device_status;        // caller's status word, or nullptr
  unsigned long long timeout_ns;
  uint64_t q, rem;           // elements per owner, and owners with one more
  uint32_t elem;             // bytes per element
  uint32_t world;
  uint32_t tmax;             // tiles of the largest owner range
  uint32_t half;             // reduce slots (and copy slots) per wave: grid / 2
  uint32_t slots;            // positions of the order: a reduce and a copy per tile
  uint32_t dst_coaligned;    // every output has the same address residue mod 16
  uint32_t drop_notify;      // test hook: 1 + flag whose notify is skipped, or 0
};

// Wait for the flag to hold the launch's epoch.  A failure of this launch is
// recorded as its epoch in the `failed` word, so an old failure never stops
// a later call.
__device__ bool na_wait(const NaArgs& a, const uint32_t* flag, uint32_t epoch) {
  const unsigned long long t0 = globaltimer();
  const unsigned long long cap = a.timeout_ns / 16ull + 4096ull;
  for (unsigned long long spin = 0;; ++spin) {
    if (ld_acquire(flag) == epoch) return true;
    if ((spin & 31ull) == 31ull) {
      if (ld_volatile(a.scratch + kNaFailed) == epoch) return false;
      if (globaltimer() - t0 > a.timeout_ns || spin > cap) {
        atomicExch(a.scratch + kNaFailed, epoch);
        return false;
      }
    }
    __nanosleep(32);
  }
}

template <typename T, int NS>
__global__ void __launch_bounds__(kNaThreads, 2) noalloc_kernel(const __grid_constant__ NaArgs a) {
  __shared__ const char* s_src[kMaxWorld];
  __shared__ char* s_dst[kMaxWorld];
  __shared__ uint64_t s_len;
  __shared__ int s_ns, s_nd, s_ok, s_kind;  // kind: 0 skip, 1 reduce, 2 copy
  __shared__ uint32_t s_flag, s_epoch;

  const uint32_t N = a.world;
  const uint32_t G = gridDim.x, c = blockIdx.x;
  if (threadIdx.x == 0) s_epoch = ld_volatile(a.scratch + kNaEpoch) + 1u;
  // Position p of the order runs on CTA p % G, in increasing p.  It is the
  // order the library's two-shot plans use, over tmax x N tiles taken
  // tile-major over the owners (an owner's missing last tile leaves its two
  // positions idle), each reduced once and then copied once: the first wave reduces
  // tiles 0 .. G-1; from the second wave on, reduce and copy positions
  // alternate in a checkerboard of (wave p / G, CTA) until the reduces run
  // out, and the rest are copies.  Copy k takes the k-th tile reduced; its
  // reduce comes at least one wave earlier (from the third wave on, two), so
  // every wait points to an earlier position.  In closed form: R, the
  // reduces before p had the reduces never run out; p reduces tile R if it
  // is a reduce position and R < tiles, else copies tile p - min(R, tiles).
  const uint64_t nt = (uint64_t)a.tmax * N;
  for (uint32_t slot = c; slot < a.slots; slot += G) {
    if (threadIdx.x == 0) {
      const uint32_t w = slot / G;
      uint64_t R = c;
      bool reduce_pos = true;
      if (w > 0) {
        R = (uint64_t)G + (uint64_t)(w - 1) * a.half + ((w & 1u) ? c / 2 : (c + 1) / 2);
        reduce_pos = ((w + c) & 1u) == 0;
      }
      const bool reduce = reduce_pos && R < nt;
      const uint64_t idx = reduce ? R : slot - (R < nt ? R : nt);
      int kind = 0;
      uint32_t o = 0;
      int64_t t = -1;
      if (idx < nt) {
        t = (int64_t)(idx / N);
        o = (uint32_t)(idx % N);
        kind = reduce ? 1 : 2;
      }
      const uint64_t olen = (a.q + (o < a.rem ? 1 : 0)) * a.elem;
      const uint64_t ostart = ((uint64_t)o * a.q + (o < a.rem ? o : a.rem)) * a.elem;
      if (kind && (uint64_t)t * kNaTile >= olen) kind = 0;
      if (kind == 2 && N == 1) kind = 0;
      int ok = 1;
      if (kind) {
        const uint64_t off = ostart + (uint64_t)t * kNaTile;
        const uint64_t rest = olen - (uint64_t)t * kNaTile;
        s_len = rest < kNaTile ? rest : kNaTile;
        s_flag = o * a.tmax + (uint32_t)t;
        if (kind == 1) {
          for (uint32_t s = 0; s < N; ++s) s_src[s] = a.in[s] + off;
          s_dst[0] = a.out[o] + off;
          s_ns = (int)N;
          s_nd = 1;
        } else {
          s_src[0] = a.out[o] + off;
          int nd = 0;
          for (uint32_t r = 0; r < N; ++r)
            if (r != o) s_dst[nd++] = a.out[r] + off;
          s_ns = 1;
          s_nd = nd;
          ok = na_wait(a, a.scratch + kNaCtlWords + s_flag, s_epoch);
        }
        if (ok && ld_volatile(a.scratch + kNaFailed) == s_epoch) ok = 0;
      }
      s_kind = kind;
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) break;
    // owner tiles with the L2 policies of the library's two-shot plans
    // (inputs evict-first, the owner tile evict-last until its copy has read
    // it, copies evict-first)
    if (s_kind == 1) {
      if (s_ns == 1)
        copy_atom<false, 2, false>(s_src[0], s_dst, 1, s_len);
      else
        reduce_owner_tile<T, NS, 1>(s_src, s_ns, s_dst, s_len);
    } else if (s_kind == 2) {
      if (a.dst_coaligned) {
        copy_owner_tile(s_src[0], s_dst, s_nd, s_len);
      } else {
        for (int j = 0; j < s_nd; ++j) copy_atom<true, 2, true>(s_src[0], s_dst + j, 1, s_len);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_kind == 1 && N > 1 && s_flag + 1 != a.drop_notify) {
      __threadfence();
      st_release(a.scratch + kNaCtlWords + s_flag, s_epoch);
    }
  }
  // The last CTA publishes the epoch.  Epochs run 1 .. 0xFFFFFFFF and start
  // again at 1: the launch that used 0xFFFFFFFF clears the flags and the
  // failure word and publishes 0, so no value of one cycle matches the next.
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.scratch + kNaDone, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  const bool wrap = s_epoch == 0xFFFFFFFFu;
  if (threadIdx.x == 0 && a.device_status)
    *a.device_status = ld_volatile(a.scratch + kNaFailed) == s_epoch ? (int)PL_ERR_TIMEOUT : (int)PL_OK;
  __syncthreads();
  if (wrap) {
    for (uint32_t i = threadIdx.x; i < (uint32_t)kNaMaxFlags; i += blockDim.x) a.scratch[kNaCtlWords + i] = 0u;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();
    a.scratch[kNaDone] = 0u;
    if (wrap) a.scratch[kNaFailed] = 0u;
    a.scratch[kNaEpoch] = wrap ? 0u : s_epoch;
    __threadfence();
  }
}

template <typename T>
const void* na_kernel(int world) {
  if (world == 8) return (const void*)noalloc_kernel<T, 8>;
  return (const void*)noalloc_kernel<T, 0>;
}

struct NaDevice {
  uint32_t* scratch = nullptr;
  int sm_count = 0;
};

std::mutex g_na_mu;
NaDevice g_na_dev[kNaMaxDevices];
// Test hook (purlin_debug_noalloc_next): settings of the next call only.
unsigned long long g_na_next_timeout_ns = 0;  // 0: the default
uint32_t g_na_next_drop = 0;                  // 1 + flag whose notify is skipped, or 0

// First call on a device: find the array's device address (host code only
// holds a stand-in for it), zero it on the stream, and note the SM count.
purlin_status na_setup(int dev, cudaStream_t stream, NaDevice* out) {
  std::lock_guard<std::mutex> lock(g_na_mu);
  NaDevice& d = g_na_dev[dev];
  if (!d.scratch) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return PL_ERR_CUDA;
    }
    if (cudaMemsetAsync(p, 0, sizeof(g_noalloc_scratch), stream) != cudaSuccess) {
      (void)cudaGetLastError();
      return PL_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
      (void)cudaGetLastError();
      return PL_ERR_CUDA;
    }
    d.sm_count = sms;
    d.scratch = (uint32_t*)p;
  }
  *out = d;
  return PL_OK;
}

}  // namespace
}  // namespace pl

extern "C" purlin_status purlin_debug_noalloc_set_epoch(uint32_t epoch, purlin_stream_t stream) {
  using namespace pl;
  // the counter holds the epoch the last launch used, 0 .. 0xFFFFFFFE: from
  // 0xFFFFFFFF the next launch would take epoch 0, the value of cleared flags
  if (epoch == 0xFFFFFFFFu) return PL_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) {
    (void)cudaGetLastError();
    return PL_ERR_CUDA;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    (void)cudaGetLastError();
    return PL_ERR_INVALID_ARG;  // a captured copy would read a dead stack slot
  }
  NaDevice d;
  if (purlin_status st = na_setup(dev, (cudaStream_t)stream, &d)) return st;
  cudaError_t e = cudaMemcpyAsync(d.scratch + kNaEpoch, &epoch, sizeof epoch, cudaMemcpyHostToDevice,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);  // `epoch` is on this stack
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PL_ERR_CUDA;
  }
  return PL_OK;
}

extern "C" purlin_status purlin_debug_noalloc_next(uint64_t timeout_ns, long long drop_tile) {
  using namespace pl;
  if (drop_tile >= (long long)kNaMaxFlags) return PL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_na_mu);
  g_na_next_timeout_ns = timeout_ns;
  g_na_next_drop = drop_tile < 0 ? 0u : (uint32_t)drop_tile + 1u;
  return PL_OK;
}

extern "C" purlin_status purlin_all_reduce_noalloc(int world, const void* const* src, void* const* dst,
                                                   size_t bytes_per_rank, purlin_dtype dtype, int* device_status,
                                                   purlin_stream_t stream) {
  using namespace pl;
  if (world < 1 || world > kMaxWorld || !src || !dst) return PL_ERR_INVALID_ARG;
  if (dtype != PL_F32 && dtype != PL_BF16) return PL_ERR_UNSUPPORTED;
  const uint64_t E = (uint64_t)elem_size(dtype);
  for (int r = 0; r < world; ++r) {
    if (!src[r] || !dst[r]) return PL_ERR_INVALID_ARG;
    if (((uintptr_t)src[r] | (uintptr_t)dst[r]) % E) return PL_ERR_ALIGNMENT;
  }
  if (bytes_per_rank % E) return PL_ERR_ALIGNMENT;
  // destinations disjoint from each other and from every source but their own (in place)
  const uintptr_t S = bytes_per_rank;
  for (int i = 0; i < world; ++i) {
    const uintptr_t d0 = (uintptr_t)dst[i], d1 = d0 + S;
    for (int j = 0; j < world; ++j) {
      const uintptr_t s0 = (uintptr_t)src[j], s1 = s0 + S;
      if (S && d0 < s1 && s0 < d1 && !(i == j && s0 == d0)) return PL_ERR_INVALID_ARG;
      if (j > i) {
        const uintptr_t e0 = (uintptr_t)dst[j], e1 = e0 + S;
        if (S && d0 < e1 && e0 < d1) return PL_ERR_INVALID_ARG;
      }
    }
  }
  const uint64_t n = bytes_per_rank / E;
  const uint64_t q = n / (uint64_t)world, rem = n % (uint64_t)world;
  const uint64_t largest = (q + (rem ? 1 : 0)) * E;
  const uint64_t tmax = (largest + kNaTile - 1) / kNaTile;
  // the fixed flag array bounds the size: world * tmax tiles of 64 KiB
  if ((uint64_t)world * tmax > (uint64_t)kNaMaxFlags) return PL_ERR_WORKSPACE;
  if (bytes_per_rank == 0) return PL_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) {
    (void)cudaGetLastError();
    return PL_ERR_CUDA;
  }
  cudaStream_t s = (cudaStream_t)stream;
  NaDevice d;
  if (purlin_status st = na_setup(dev, s, &d)) return st;

  const void* fn = dtype == PL_F32 ? na_kernel<float>(world) : na_kernel<bf16_tag>(world);
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kNaThreads, 0) != cudaSuccess || occ < 1) {
    (void)cudaGetLastError();
    return PL_ERR_LAUNCH;
  }
  NaArgs a = {};
  uint32_t same = 1;
  for (int r = 0; r < world; ++r) {
    a.in[r] = (const char*)src[r];
    a.out[r] = (char*)dst[r];
    if ((((uintptr_t)dst[r]) & 15u) != (((uintptr_t)dst[0]) & 15u)) same = 0;
  }
  int ctas = std::min(occ, 2) * d.sm_count;
  a.scratch = d.scratch;
  a.device_status = device_status;
  a.timeout_ns = 2000000000ull;
  {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (g_na_next_timeout_ns) a.timeout_ns = g_na_next_timeout_ns;
    a.drop_notify = g_na_next_drop;
    g_na_next_timeout_ns = 0;
    g_na_next_drop = 0;
  }
  a.q = q;
  a.rem = rem;
  a.elem = (uint32_t)E;
  a.world = (uint32_t)world;
  a.tmax = (uint32_t)tmax;
  // an even grid (the checkerboard of positions), no larger than two positions per tile
  const uint64_t nt = tmax * (uint64_t)world;
  uint64_t g = std::min<uint64_t>((uint64_t)ctas, 2 * nt);
  g = std::max<uint64_t>(2, g & ~1ull);
  a.half = (uint32_t)(g / 2);
  a.slots = (uint32_t)(2 * nt);
  a.dst_coaligned = same;
  const int grid = (int)g;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kNaThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the CTAs wait on each other: all must be resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    (void)cudaGetLastError();
    return PL_ERR_LAUNCH;
  }
  return PL_OK;
}
