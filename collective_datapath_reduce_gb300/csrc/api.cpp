// C ABI of the datapath: handle, workspace, argument checks, plan cache and
// launch.  Every data movement happens in the kernels of kernels_*.cu; this
// file only validates, plans and launches.
//
// Purlin 0.6.5 (PyPI page), "Host-side": create one context per communicator
// with a workspace of staging and signal buffers, run collectives on a
// stream, finalize after the last one.  Here the context owns the SNAC flag
// array and a status word, and caches one plan per call shape.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "kargs.h"
#include "plan.h"
#include "purlin_gb.h"

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
// Library-owned workspace: flags for the two-shot and ring AllReduce layouts
// at the table's tile sizes up to several GiB per rank (8 MiB of flags).
constexpr size_t kDefaultFlags = PURLIN_DEFAULT_WORKSPACE_FLAGS;

struct DevPlan {
  pl::Plan plan;
  const void* fn = nullptr;
  int threads = 0;
  int smem = 0;              // dynamic shared memory (bulk path ring)
  uint32_t ring_chunk = 0;   // bulk path: bytes per source tile in a slot
  void* d_mem = nullptr;     // items, then cta_begin
  void* h_mem = nullptr;     // pinned host copy (kept: a captured upload replays from it)
  size_t bytes = 0;
  const pl::Item* d_items = nullptr;
  const uint32_t* d_cta = nullptr;
  bool uploaded = false;
};

}  // namespace

struct purlin_ctx {
  int world = 0;
  int device = 0;
  int sm_count = 0;
  int arch = 0;
  int max_ctas_per_sm = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  bool ws_owned = false;
  int ws_grown = 0;             // times the library-owned workspace was enlarged
  uint32_t* ctl = nullptr;
  uint32_t* flags = nullptr;
  size_t flag_cap = 0;
  std::mutex mu;
  std::unordered_map<std::string, std::unique_ptr<DevPlan>> plans;
  pl::Tune over;
  bool has_over = false;
  unsigned long long timeout_ns = kDefaultTimeoutNs;
  long long drop_notify = -1;
  int limit_side = -1, limit_rank = 0;  // purlin_debug_limit_buffer, for the next launch
  uint64_t limit_bytes = 0;
  unsigned long long* trace = nullptr;  // caller's trace buffer, or nullptr
  uint32_t trace_cap = 0;
  bool finalized = false;
};

namespace {

purlin_status cuda_fail(cudaError_t e) {
  (void)cudaGetLastError();  // clear the sticky-free error state
  return e == cudaSuccess ? PL_OK : PL_ERR_CUDA;
}

void free_plan(DevPlan* d) {
  if (d->d_mem) cudaFree(d->d_mem);
  if (d->h_mem) cudaFreeHost(d->h_mem);
  d->d_mem = d->h_mem = nullptr;
}

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return st != cudaStreamCaptureStatusNone;
}

// Largest dynamic shared memory a CTA may use on sm_100-class GPUs (227 KiB),
// less room for the kernels' static shared memory.
constexpr int kMaxDynSmem = 227 * 1024 - 1024;

const void* pick_kernel(const pl::Plan& p) {
  if (p.tune.path == pl::kPathBulk) {
    if (p.nsrc <= 1) return p.tune.schedule == pl::kSchedItem ? pl::kernel_bulk_copy() : pl::kernel_stream_copy();
    if (p.dtype == pl::kF32) return pl::kernel_bulk_reduce_f32(p.nsrc);
    if (p.dtype == pl::kBF16) return pl::kernel_bulk_reduce_bf16(p.nsrc);
    return nullptr;
  }
  if (p.nsrc <= 1) {
    int u = p.tune.unroll;
    u = u >= 8 ? 8 : u >= 4 ? 4 : u >= 2 ? 2 : 1;
    return pl::kernel_copy(u);
  }
  if (p.tune.store_hint == 3) {
    if (p.dtype == pl::kF32) return pl::kernel_reduce_l2_f32(p.nsrc, p.tune.unroll);
    if (p.dtype == pl::kBF16) return pl::kernel_reduce_l2_bf16(p.nsrc, p.tune.unroll);
    return nullptr;
  }
  if (p.tune.layout == pl::kRing && p.sync) {
    if (p.dtype == pl::kF32) return pl::kernel_reduce_ring_f32(p.tune.unroll);
    if (p.dtype == pl::kBF16) return pl::kernel_reduce_ring_bf16(p.tune.unroll);
    return nullptr;
  }
  if (p.dtype == pl::kF32) return pl::kernel_reduce_f32(p.nsrc, p.tune.unroll);
  if (p.dtype == pl::kBF16) return pl::kernel_reduce_bf16(p.nsrc, p.tune.unroll);
  return nullptr;
}

struct Range {
  uintptr_t lo, hi;
};

bool overlaps(const Range& a, const Range& b) {
  return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// Destinations must be pairwise disjoint and must not overlap any source,
// except an exact in-place pair src[r] == dst[r] when allowed.  A buffer whose
// end would pass the top of the address space is refused too.
purlin_status check_overlap(const std::vector<Range>& src, const std::vector<Range>& dst,
                            bool allow_in_place) {
  for (const Range& r : src)
    if (r.hi < r.lo) return PL_ERR_INVALID_ARG;
  for (const Range& r : dst)
    if (r.hi < r.lo) return PL_ERR_INVALID_ARG;
  for (size_t i = 0; i < dst.size(); ++i) {
    for (size_t j = i + 1; j < dst.size(); ++j)
      if (overlaps(dst[i], dst[j])) return PL_ERR_INVALID_ARG;
    for (size_t s = 0; s < src.size(); ++s) {
      if (!overlaps(dst[i], src[s])) continue;
      if (allow_in_place && s == i && src[s].lo == dst[i].lo && src[s].hi == dst[i].hi) continue;
      return PL_ERR_INVALID_ARG;
    }
  }
  return PL_OK;
}

purlin_status ensure_flags(purlin_ctx* h, size_t need, cudaStream_t stream) {
  if (need <= h->flag_cap) return PL_OK;
  if (!h->ws_owned) return PL_ERR_WORKSPACE;
  if (capturing(stream)) return PL_ERR_WORKSPACE;
  size_t cap = std::max(need, h->flag_cap * 2);
  size_t bytes = pl::kCtlBytes + cap * sizeof(uint32_t);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  void* nws = nullptr;
  if ((e = cudaMalloc(&nws, bytes)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemset(nws, 0, bytes)) != cudaSuccess) {
    cudaFree(nws);
    return cuda_fail(e);
  }
  // keep a pending device error across the move
  uint32_t status = 0;
  cudaMemcpy(&status, h->ctl, sizeof(status), cudaMemcpyDeviceToHost);
  cudaMemcpy(nws, &status, sizeof(status), cudaMemcpyHostToDevice);
  cudaFree(h->ws);
  h->ws = nws;
  h->ws_bytes = bytes;
  h->ws_grown += 1;
  h->ctl = (uint32_t*)nws;
  h->flags = (uint32_t*)((char*)nws + pl::kCtlBytes);
  h->flag_cap = cap;
  return PL_OK;
}

std::string plan_key(int coll, int world, int dtype, const uint64_t* sizes, size_t n,
                     const uint8_t* sres, const uint8_t* dres, bool host_mem, const purlin_ctx* h) {
  std::string k;
  k.reserve(64 + n * 8);
  auto put = [&](const void* p, size_t b) { k.append((const char*)p, b); };
  put(&host_mem, sizeof host_mem);
  put(&coll, sizeof coll);
  put(&world, sizeof world);
  put(&dtype, sizeof dtype);
  put(sizes, n * sizeof(uint64_t));
  put(sres, (size_t)world);
  put(dres, (size_t)world);
  if (h->has_over) put(&h->over, sizeof h->over);
  return k;
}

purlin_status get_plan(purlin_ctx* h, int coll, int world, int dtype, const uint64_t* sizes, size_t n,
                       const uint8_t* sres, const uint8_t* dres, bool host_mem, cudaStream_t stream,
                       DevPlan** out) {
  const std::string key = plan_key(coll, world, dtype, sizes, n, sres, dres, host_mem, h);
  auto it = h->plans.find(key);
  if (it != h->plans.end()) {
    *out = it->second.get();
    return PL_OK;
  }
  auto d = std::make_unique<DevPlan>();
  pl::Tune over = h->has_over ? h->over : pl::Tune{};
  if (host_mem) {
    // buffers in host memory: register path, item by item (the bulk copy
    // engines are kept to device memory)
    over.path = pl::kPathRegister;
    over.schedule = pl::kSchedItem;
  }
  int st = pl::build_plan(coll, world, dtype, sizes, n, sres, dres, h->sm_count, 0, over, &d->plan);
  if (st) return (purlin_status)st;
  d->fn = pick_kernel(d->plan);
  if (!d->fn) return PL_ERR_UNSUPPORTED;
  d->threads = d->plan.tune.threads;
  if (d->plan.tune.path == pl::kPathBulk) {
    // dynamic shared memory this kernel can take: the per-block opt-in limit
    // less its static shared memory (and never more than kMaxDynSmem)
    int max_dyn = kMaxDynSmem;
    {
      cudaFuncAttributes fa;
      int optin = 0;
      cudaError_t e = cudaFuncGetAttributes(&fa, d->fn);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device);
      if (e != cudaSuccess) return cuda_fail(e);
      max_dyn = std::min(max_dyn, optin - (int)fa.sharedSizeBytes);
    }
    // Ring of `stages` slots.  A reduce slot holds nsrc input tiles and one
    // output tile.  A copy slot holds one chunk, or, for sources that are not
    // 16-byte aligned, a source window of chunk + 16 bytes; two output tiles
    // of one chunk each follow the copy slots (the shifted copy cuts its
    // destination vectors into them).  A reduce ring is always at least as
    // large as that copy layout, so a reduce plan's copy items fit too.
    const bool copy_ring = d->plan.nsrc <= 1;
    const int tiles = copy_ring ? 1 : d->plan.nsrc + 1;
    const int stages = d->plan.tune.stages;
    int64_t ch = d->plan.tune.chunk_bytes;
    const int64_t fit = copy_ring ? (max_dyn - 16 * stages) / (stages + 2) : (max_dyn / stages - 16) / tiles;
    if (ch > fit) ch = fit;
    const int64_t tx_cap = copy_ring ? (1 << 20) / 2 : (1 << 20) / tiles;
    if (ch > tx_cap) ch = tx_cap;  // mbarrier transaction count stays below 2^20
    ch &= ~(int64_t)15;
    if (ch < 16) return PL_ERR_INVALID_ARG;
    d->ring_chunk = (uint32_t)ch;
    d->smem = copy_ring ? (int)(stages * (ch + 16) + 2 * ch) : (int)(stages * (tiles * ch + 16));
    // The limit is a property of the kernel function, shared by every plan that
    // launches it: raise it to the largest ring any plan may use, never lower it.
    cudaError_t e = cudaFuncSetAttribute(d->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (d->plan.sync) {
    // CTAs of this plan wait on each other: all of them must be resident.
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, d->fn, d->threads, d->smem);
    if (e != cudaSuccess) return cuda_fail(e);
    if (occ < 1) return PL_ERR_LAUNCH;
    if (d->plan.grid > occ * h->sm_count) {
      st = pl::build_plan(coll, world, dtype, sizes, n, sres, dres, h->sm_count, occ, over, &d->plan);
      if (st) return (purlin_status)st;
    }
  }
  const std::string bad = pl::check_plan(d->plan);
  if (!bad.empty()) return PL_ERR_INVALID_ARG;
  const size_t ib = d->plan.items.size() * sizeof(pl::Item);
  const size_t cb = d->plan.cta_begin.size() * sizeof(uint32_t);
  d->bytes = ib + cb;
  if (d->bytes) {
    cudaError_t e = cudaMalloc(&d->d_mem, d->bytes);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMallocHost(&d->h_mem, d->bytes);
    if (e != cudaSuccess) {
      free_plan(d.get());
      return cuda_fail(e);
    }
    if (ib) std::memcpy(d->h_mem, d->plan.items.data(), ib);
    if (cb) std::memcpy((char*)d->h_mem + ib, d->plan.cta_begin.data(), cb);
    if (capturing(stream)) {
      e = cudaMemcpyAsync(d->d_mem, d->h_mem, d->bytes, cudaMemcpyHostToDevice, stream);
    } else {
      e = cudaMemcpy(d->d_mem, d->h_mem, d->bytes, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
      free_plan(d.get());
      return cuda_fail(e);
    }
    d->d_items = (const pl::Item*)d->d_mem;
    d->d_cta = cb ? (const uint32_t*)((char*)d->d_mem + ib) : nullptr;
  }
  *out = d.get();
  h->plans.emplace(key, std::move(d));
  return PL_OK;
}

// Plan (cached) and launch one call.  in/out: `nin` / `nout` buffer pointers.
// Where one rank buffer lives, and the address the kernel uses for it.
// Device and managed memory take every path.  Host memory the device maps
// (cudaHostAlloc, cudaHostRegister) is read and written in place over the
// host link.  Anything else is refused: another device's memory, and any
// address the driver does not know -- even where the device could reach
// pageable memory, an unknown address may not be a mapping at all, and the
// kernel would fault on it.
purlin_status locate(const purlin_ctx* h, const void* p, const void** dev_p, bool* host) {
  *dev_p = p;
  if (!p) return PL_OK;  // a zero-byte rank of a V collective
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PL_ERR_INVALID_ARG;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
      return at.device == h->device ? PL_OK : PL_ERR_INVALID_ARG;
    case cudaMemoryTypeManaged:
      return PL_OK;
    case cudaMemoryTypeHost:
      if (at.devicePointer) *dev_p = at.devicePointer;
      *host = true;
      return PL_OK;
    default:  // unregistered: pageable host memory, or no mapping at all
      return PL_ERR_INVALID_ARG;
  }
}

purlin_status run(purlin_ctx* h, int coll, int world, int dtype, const uint64_t* sizes, size_t n,
                  const void* const* in_arg, int nin, void* const* out_arg, int nout, cudaStream_t stream) {
  // The workspace and the plans live on the device that was current when the
  // handle was created; launching with another device current would hand the
  // kernel pointers of a different GPU.
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return cuda_fail(cudaErrorInvalidDevice);
  if (cur != h->device) return PL_ERR_INVALID_ARG;
  const void* in[pl::kMaxWorld] = {};
  void* out[pl::kMaxWorld] = {};
  bool host_mem = false;
  purlin_status st;
  for (int r = 0; r < nin; ++r)
    if ((st = locate(h, in_arg[r], &in[r], &host_mem))) return st;
  for (int r = 0; r < nout; ++r) {
    const void* q = nullptr;
    if ((st = locate(h, out_arg[r], &q, &host_mem))) return st;
    out[r] = const_cast<void*>(q);
  }
  uint8_t sres[pl::kMaxWorld] = {}, dres[pl::kMaxWorld] = {};
  for (int r = 0; r < nin; ++r) sres[r] = (uint8_t)((uintptr_t)in[r] & 15u);
  for (int r = 0; r < nout; ++r) dres[r] = (uint8_t)((uintptr_t)out[r] & 15u);
  std::lock_guard<std::mutex> lock(h->mu);
  DevPlan* d = nullptr;
  st = get_plan(h, coll, world, dtype, sizes, n, sres, dres, host_mem, stream, &d);
  if (st) return st;
  if (d->plan.items.empty()) return PL_OK;
  if ((st = ensure_flags(h, (size_t)d->plan.n_flags, stream))) return st;

  pl::KArgs a;
  std::memset(&a, 0, sizeof a);
  for (int r = 0; r < nin; ++r) a.in[r] = (const char*)in[r];
  for (int r = 0; r < nout; ++r) a.out[r] = (char*)out[r];
  a.items = d->d_items;
  a.cta_begin = d->d_cta;
  a.n_items = (uint32_t)d->plan.items.size();
  a.strided = d->plan.strided ? 1u : 0u;
  a.sync = d->plan.sync ? 1u : 0u;
  a.queue = d->plan.queue ? 1u : 0u;
  a.flags = h->flags;
  a.ctl = h->ctl;
  a.timeout_ns = h->timeout_ns;
  a.drop_notify = h->drop_notify >= 0 ? (uint32_t)(h->drop_notify + 1) : 0u;
  a.nsrc = d->plan.nsrc;
  a.store_hint = d->plan.tune.store_hint;
  a.stages = d->plan.tune.stages;
  a.chunk_bytes = d->ring_chunk;
  a.trace = h->trace;
  a.trace_cap = h->trace_cap;
  a.flag_cap = (uint32_t)std::min<size_t>(h->flag_cap, 0xFFFFFFFFu);
  h->drop_notify = -1;
  for (int r = 0; r < pl::kMaxWorld; ++r) {
    a.in_bytes[r] = d->plan.in_bytes[r];
    a.out_bytes[r] = d->plan.out_bytes[r];
  }
  if (h->limit_side >= 0) {
    uint64_t* b = h->limit_side ? a.out_bytes : a.in_bytes;
    b[h->limit_rank] = std::min<uint64_t>(b[h->limit_rank], h->limit_bytes);
    h->limit_side = -1;
  }

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)d->plan.grid);
  cfg.blockDim = dim3((unsigned)d->threads);
  cfg.dynamicSmemBytes = (size_t)d->smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (d->plan.sync) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    // programmatic dependent launch: the launch may start once the previous
    // kernel on the stream has retired its CTAs; the kernel waits for that
    // grid's completion (grid_dep_wait) before it touches memory
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, d->fn, args);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PL_ERR_LAUNCH;
  }
  return PL_OK;
}

// Handles the library created and has not finalized, and the addresses of
// finalized ones, so that a call on a finalized handle reports it instead of
// touching freed memory.
std::mutex g_reg_mu;
std::unordered_set<const purlin_ctx*> g_live, g_dead;

purlin_status check_handle(purlin_ctx* h) {
  if (!h) return PL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_reg_mu);
  if (g_live.count(h)) return PL_OK;
  return g_dead.count(h) ? PL_ERR_FINALIZED : PL_ERR_INVALID_ARG;
}

purlin_status check_ptrs(const void* const* p, int n) {
  if (!p) return PL_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!p[i]) return PL_ERR_INVALID_ARG;
  return PL_OK;
}

// Pointers may be NULL only where the rank's buffer holds zero bytes.
purlin_status check_ptrs_sized(const void* const* p, int n, const std::vector<uint64_t>& bytes) {
  if (!p) return PL_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!p[i] && bytes[(size_t)i]) return PL_ERR_INVALID_ARG;
  return PL_OK;
}

purlin_status check_reduce_args(purlin_dtype dtype, purlin_mode mode) {
  if (mode != PL_DETERMINISTIC) return PL_ERR_UNSUPPORTED;
  if (dtype != PL_F32 && dtype != PL_BF16) return PL_ERR_UNSUPPORTED;
  return PL_OK;
}

purlin_status check_elem_aligned(const void* const* p, int n, size_t e) {
  for (int i = 0; i < n; ++i)
    if ((uintptr_t)p[i] % e) return PL_ERR_ALIGNMENT;
  return PL_OK;
}

// a + b, or false where the sum does not fit in 64 bits
bool add_u64(uint64_t a, uint64_t b, uint64_t* sum) { return !__builtin_add_overflow(a, b, sum); }

std::vector<Range> ranges(const void* const* p, int n, const std::vector<uint64_t>& bytes) {
  std::vector<Range> r((size_t)n);
  for (int i = 0; i < n; ++i) r[i] = Range{(uintptr_t)p[i], (uintptr_t)p[i] + (uintptr_t)bytes[i]};
  return r;
}

}  // namespace

extern "C" {

size_t purlin_workspace_bytes(int world, size_t max_bytes_per_rank) {
  if (world < 1 || world > PURLIN_MAX_WORLD) return 0;
  // flags of the SNAC AllReduce layouts at the table's tile size, for the
  // smallest element (bf16): one per tile of each rank's share (two-shot), or
  // one per tile and stage but the last of 2 (world - 1) stages (ring)
  const uint64_t S = max_bytes_per_rank;
  const pl::Tune t = pl::tune_table(pl::kAllReduce, world, pl::kBF16, S);
  // ring: its tiles are a 64th of a rank's share, at least 64 KiB
  const pl::Tune tr = pl::resolve_tune(pl::kAllReduce, pl::kAllReduce, world, pl::kBF16, S,
                                       [] { pl::Tune o; o.layout = pl::kRing; return o; }());
  const uint64_t per_owner = (S / 2 + (uint64_t)world - 1) / (uint64_t)world * 2;
  const uint64_t ring_tiles = std::max<uint64_t>(1, (per_owner + (uint64_t)tr.chunk_bytes - 1) / (uint64_t)tr.chunk_bytes);
  const uint64_t per_tile = world > 1 ? 2 * (uint64_t)world - 3 : 1;
  const uint64_t ring = (uint64_t)world * ring_tiles * per_tile;
  // two-shot: one flag per tile of each owner's share
  const uint64_t two_shot = (uint64_t)world * std::max<uint64_t>(1, (per_owner + (uint64_t)t.chunk_bytes - 1) /
                                                                       (uint64_t)t.chunk_bytes);
  return (size_t)pl::kCtlBytes + (size_t)std::max(ring, two_shot) * sizeof(uint32_t);
}

purlin_status purlin_initialize(int world, void* workspace, size_t workspace_bytes, purlin_stream_t stream,
                                purlin_handle* out) {
  if (!out) return PL_ERR_INVALID_ARG;
  *out = nullptr;
  if (world < 1 || world > PURLIN_MAX_WORLD) return PL_ERR_INVALID_ARG;
  if (workspace && (workspace_bytes < (size_t)pl::kCtlBytes || ((uintptr_t)workspace & 255u)))
    return PL_ERR_WORKSPACE;
  auto h = std::make_unique<purlin_ctx>();
  h->world = world;
  cudaError_t e;
  if ((e = cudaGetDevice(&h->device)) != cudaSuccess) return cuda_fail(e);
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device)) != cudaSuccess)
    return cuda_fail(e);
  h->arch = major * 10 + minor;
  const void* probe = pl::kernel_reduce_bf16(8, 1);
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&h->max_ctas_per_sm, probe, 512, 0)) != cudaSuccess)
    return cuda_fail(e);
  cudaStream_t s = (cudaStream_t)stream;
  if (workspace) {
    h->ws = workspace;
    h->ws_bytes = workspace_bytes;
    h->ws_owned = false;
  } else {
    // NULL workspace: the library allocates the default, or workspace_bytes if larger
    h->ws_bytes = std::max(workspace_bytes, pl::kCtlBytes + kDefaultFlags * sizeof(uint32_t));
    if ((e = cudaMalloc(&h->ws, h->ws_bytes)) != cudaSuccess) return cuda_fail(e);
    h->ws_owned = true;
  }
  h->ctl = (uint32_t*)h->ws;
  h->flags = (uint32_t*)((char*)h->ws + pl::kCtlBytes);
  h->flag_cap = (h->ws_bytes - pl::kCtlBytes) / sizeof(uint32_t);
  if ((e = cudaMemsetAsync(h->ws, 0, h->ws_bytes, s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess) {
    if (h->ws_owned) cudaFree(h->ws);
    return cuda_fail(e);
  }
  {
    std::lock_guard<std::mutex> lock(g_reg_mu);
    g_dead.erase(h.get());
    g_live.insert(h.get());
  }
  *out = h.release();
  return PL_OK;
}

purlin_status purlin_finalize(purlin_handle h, purlin_stream_t stream) {
  if (purlin_status st = check_handle(h)) return st;
  {
    std::lock_guard<std::mutex> lock(g_reg_mu);
    g_live.erase(h);
    g_dead.insert(h);
  }
  purlin_status result = PL_OK;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) result = cuda_fail(e);
  uint32_t status = 0;
  if (cudaMemcpy(&status, h->ctl, sizeof status, cudaMemcpyDeviceToHost) == cudaSuccess && status)
    result = (purlin_status)status;
  for (auto& kv : h->plans) free_plan(kv.second.get());
  h->plans.clear();
  if (h->ws_owned && h->ws) cudaFree(h->ws);
  h->ws = nullptr;
  h->finalized = true;
  delete h;
  return result;
}

purlin_status purlin_all_reduce(purlin_handle h, const void* const* src, void* const* dst,
                                size_t bytes_per_rank, purlin_dtype dtype, purlin_mode mode,
                                purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h)) || (st = check_reduce_args(dtype, mode))) return st;
  const int N = h->world;
  if ((st = check_ptrs(src, N)) || (st = check_ptrs((const void* const*)dst, N))) return st;
  const size_t E = (size_t)pl::elem_size(dtype);
  if (bytes_per_rank % E) return PL_ERR_ALIGNMENT;
  if ((st = check_elem_aligned(src, N, E)) || (st = check_elem_aligned((const void* const*)dst, N, E)))
    return st;
  if (bytes_per_rank == 0) return PL_OK;
  std::vector<uint64_t> b((size_t)N, bytes_per_rank);
  if ((st = check_overlap(ranges(src, N, b), ranges((const void* const*)dst, N, b), true))) return st;
  const uint64_t sz = bytes_per_rank;
  return run(h, pl::kAllReduce, N, dtype, &sz, 1, src, N, dst, N, (cudaStream_t)stream);
}

purlin_status purlin_reduce_scatter(purlin_handle h, const void* const* src, void* const* dst,
                                    size_t in_bytes_per_rank, purlin_dtype dtype, purlin_mode mode,
                                    purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h)) || (st = check_reduce_args(dtype, mode))) return st;
  const int N = h->world;
  if ((st = check_ptrs(src, N)) || (st = check_ptrs((const void* const*)dst, N))) return st;
  const size_t E = (size_t)pl::elem_size(dtype);
  if (in_bytes_per_rank % E) return PL_ERR_ALIGNMENT;
  if ((in_bytes_per_rank / E) % (size_t)N) return PL_ERR_INVALID_ARG;
  if ((st = check_elem_aligned(src, N, E)) || (st = check_elem_aligned((const void* const*)dst, N, E)))
    return st;
  if (in_bytes_per_rank == 0) return PL_OK;
  std::vector<uint64_t> bi((size_t)N, in_bytes_per_rank), bo((size_t)N, in_bytes_per_rank / N);
  if ((st = check_overlap(ranges(src, N, bi), ranges((const void* const*)dst, N, bo), false))) return st;
  const uint64_t sz = in_bytes_per_rank;
  return run(h, pl::kReduceScatter, N, dtype, &sz, 1, src, N, dst, N, (cudaStream_t)stream);
}

purlin_status purlin_reduce_scatter_v(purlin_handle h, const void* const* src, void* const* dst,
                                      const size_t* bytes, purlin_dtype dtype, purlin_mode mode,
                                      purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h)) || (st = check_reduce_args(dtype, mode))) return st;
  const int N = h->world;
  if (!bytes) return PL_ERR_INVALID_ARG;
  const size_t E = (size_t)pl::elem_size(dtype);
  std::vector<uint64_t> sz((size_t)N), bi((size_t)N);
  uint64_t total = 0;
  for (int r = 0; r < N; ++r) {
    if (bytes[r] % E) return PL_ERR_ALIGNMENT;
    sz[r] = bytes[r];
    if (!add_u64(total, bytes[r], &total)) return PL_ERR_INVALID_ARG;
  }
  std::fill(bi.begin(), bi.end(), total);
  if ((st = check_ptrs_sized(src, N, bi)) || (st = check_ptrs_sized((const void* const*)dst, N, sz))) return st;
  if ((st = check_elem_aligned(src, N, E)) || (st = check_elem_aligned((const void* const*)dst, N, E)))
    return st;
  if (total == 0) return PL_OK;
  if ((st = check_overlap(ranges(src, N, bi), ranges((const void* const*)dst, N, sz), false))) return st;
  return run(h, pl::kReduceScatterV, N, dtype, sz.data(), sz.size(), src, N, dst, N, (cudaStream_t)stream);
}

purlin_status purlin_all_gather(purlin_handle h, const void* const* src, void* const* dst,
                                size_t in_bytes_per_rank, purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  const int N = h->world;
  if ((st = check_ptrs(src, N)) || (st = check_ptrs((const void* const*)dst, N))) return st;
  if (in_bytes_per_rank == 0) return PL_OK;
  if (in_bytes_per_rank > UINT64_MAX / (uint64_t)N) return PL_ERR_INVALID_ARG;  // outputs of world x bytes
  std::vector<uint64_t> bi((size_t)N, in_bytes_per_rank), bo((size_t)N, in_bytes_per_rank * N);
  if ((st = check_overlap(ranges(src, N, bi), ranges((const void* const*)dst, N, bo), false))) return st;
  const uint64_t sz = in_bytes_per_rank;
  return run(h, pl::kAllGather, N, pl::kU8, &sz, 1, src, N, dst, N, (cudaStream_t)stream);
}

purlin_status purlin_all_to_all(purlin_handle h, const void* const* src, void* const* dst,
                                size_t bytes_per_rank, purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  const int N = h->world;
  if ((st = check_ptrs(src, N)) || (st = check_ptrs((const void* const*)dst, N))) return st;
  if (bytes_per_rank % (size_t)N) return PL_ERR_INVALID_ARG;
  if (bytes_per_rank == 0) return PL_OK;
  std::vector<uint64_t> b((size_t)N, bytes_per_rank);
  if ((st = check_overlap(ranges(src, N, b), ranges((const void* const*)dst, N, b), false))) return st;
  const uint64_t sz = bytes_per_rank;
  return run(h, pl::kAllToAll, N, pl::kU8, &sz, 1, src, N, dst, N, (cudaStream_t)stream);
}

purlin_status purlin_all_gather_v(purlin_handle h, const void* const* src, void* const* dst,
                                  const size_t* bytes, purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  const int N = h->world;
  if (!bytes) return PL_ERR_INVALID_ARG;
  std::vector<uint64_t> sz((size_t)N), bo((size_t)N);
  uint64_t total = 0;
  for (int r = 0; r < N; ++r) {
    sz[r] = bytes[r];
    if (!add_u64(total, bytes[r], &total)) return PL_ERR_INVALID_ARG;
  }
  std::fill(bo.begin(), bo.end(), total);
  if ((st = check_ptrs_sized(src, N, sz)) || (st = check_ptrs_sized((const void* const*)dst, N, bo))) return st;
  if (total == 0) return PL_OK;
  if ((st = check_overlap(ranges(src, N, sz), ranges((const void* const*)dst, N, bo), false))) return st;
  return run(h, pl::kAllGatherV, N, pl::kU8, sz.data(), sz.size(), src, N, dst, N, (cudaStream_t)stream);
}

purlin_status purlin_all_to_all_v(purlin_handle h, const void* const* src, void* const* dst,
                                  const size_t* bytes, purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  const int N = h->world;
  if (!bytes) return PL_ERR_INVALID_ARG;
  std::vector<uint64_t> sz((size_t)N * N), bi((size_t)N, 0), bo((size_t)N, 0);
  uint64_t total = 0;
  for (int s = 0; s < N; ++s)
    for (int d = 0; d < N; ++d) {
      const uint64_t c = bytes[(size_t)s * N + d];
      sz[(size_t)s * N + d] = c;
      if (!add_u64(bi[s], c, &bi[s]) || !add_u64(bo[d], c, &bo[d]) || !add_u64(total, c, &total))
        return PL_ERR_INVALID_ARG;
    }
  if ((st = check_ptrs_sized(src, N, bi)) || (st = check_ptrs_sized((const void* const*)dst, N, bo))) return st;
  if (total == 0) return PL_OK;
  if ((st = check_overlap(ranges(src, N, bi), ranges((const void* const*)dst, N, bo), false))) return st;
  return run(h, pl::kAllToAllV, N, pl::kU8, sz.data(), sz.size(), src, N, dst, N, (cudaStream_t)stream);
}

purlin_status purlin_atom_copy(purlin_handle h, const void* src, void* const* dst, int ndst, size_t bytes,
                               purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  if (!src || ndst < 1 || ndst > PURLIN_MAX_WORLD) return PL_ERR_INVALID_ARG;
  if ((st = check_ptrs((const void* const*)dst, ndst))) return st;
  if (bytes == 0) return PL_OK;
  const void* srcs[1] = {src};
  std::vector<uint64_t> bi(1, bytes), bo((size_t)ndst, bytes);
  if ((st = check_overlap(ranges(srcs, 1, bi), ranges((const void* const*)dst, ndst, bo), false))) return st;
  const uint64_t sz = bytes;
  return run(h, pl::kAtomCopy, ndst, pl::kU8, &sz, 1, srcs, 1, dst, ndst, (cudaStream_t)stream);
}

purlin_status purlin_atom_reduce(purlin_handle h, const void* const* src, int nsrc, void* const* dst,
                                 int ndst, size_t bytes, purlin_dtype dtype, purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h)) || (st = check_reduce_args(dtype, PL_DETERMINISTIC))) return st;
  if (nsrc < 1 || nsrc > PURLIN_MAX_WORLD || ndst < 1 || ndst > PURLIN_MAX_WORLD) return PL_ERR_INVALID_ARG;
  if ((st = check_ptrs(src, nsrc)) || (st = check_ptrs((const void* const*)dst, ndst))) return st;
  const size_t E = (size_t)pl::elem_size(dtype);
  if (bytes % E) return PL_ERR_ALIGNMENT;
  if ((st = check_elem_aligned(src, nsrc, E)) || (st = check_elem_aligned((const void* const*)dst, ndst, E)))
    return st;
  if (bytes == 0) return PL_OK;
  std::vector<uint64_t> bi((size_t)nsrc, bytes), bo((size_t)ndst, bytes);
  if ((st = check_overlap(ranges(src, nsrc, bi), ranges((const void* const*)dst, ndst, bo), false))) return st;
  const uint64_t sz[3] = {bytes, (uint64_t)nsrc, (uint64_t)ndst};
  return run(h, pl::kAtomReduce, std::max(nsrc, ndst), dtype, sz, 3, src, nsrc, dst, ndst,
             (cudaStream_t)stream);
}

purlin_status purlin_status_get(purlin_handle h, purlin_stream_t stream, int* device_status) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  if (!device_status) return PL_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t v = 0;
  if ((e = cudaMemcpy(&v, h->ctl, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  if (v) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpy(h->ctl, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e);
  }
  *device_status = (int)v;
  return PL_OK;
}

const char* purlin_status_string(purlin_status s) {
  switch (s) {
    case PL_OK: return "ok";
    case PL_ERR_INVALID_ARG: return "invalid argument";
    case PL_ERR_ALIGNMENT: return "pointer or size not aligned to the element size";
    case PL_ERR_UNSUPPORTED: return "unsupported dtype, mode or layout";
    case PL_ERR_WORKSPACE: return "workspace too small";
    case PL_ERR_CUDA: return "CUDA runtime error";
    case PL_ERR_LAUNCH: return "kernel launch failed";
    case PL_ERR_TIMEOUT: return "a SNAC wait on the device ran out of time";
    case PL_ERR_FINALIZED: return "handle already finalized";
    case PL_ERR_BOUNDS: return "a work item reached outside a rank buffer (checking build)";
  }
  return "unknown status";
}

purlin_status purlin_tune_get(purlin_handle h, purlin_coll coll, purlin_dtype dtype, size_t bytes_per_rank,
                              purlin_tune* out) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  if (!out) return PL_ERR_INVALID_ARG;
  const pl::Tune over = h->has_over ? h->over : pl::Tune{};
  pl::Tune t = pl::resolve_tune(coll, coll, h->world, dtype, bytes_per_rank, over);
  const bool reduce = coll == PL_COLL_ALL_REDUCE || coll == PL_COLL_REDUCE_SCATTER ||
                      coll == PL_COLL_REDUCE_SCATTER_V;
  if (t.path == pl::kPathRegister && reduce && h->world > 8) t.threads = std::min(t.threads, 256);
  static_assert(sizeof(pl::Tune) == sizeof(purlin_tune), "tune layout");
  std::memcpy(out, &t, sizeof t);
  return PL_OK;
}

purlin_status purlin_tune_override(purlin_handle h, const purlin_tune* t) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  std::lock_guard<std::mutex> lock(h->mu);
  if (!t) {
    h->has_over = false;
    h->over = pl::Tune{};
  } else {
    std::memcpy(&h->over, t, sizeof h->over);
    h->has_over = true;
  }
  return PL_OK;
}

purlin_status purlin_set_wait_timeout_ns(purlin_handle h, uint64_t ns) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  if (ns == 0) return PL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(h->mu);
  h->timeout_ns = ns;
  return PL_OK;
}

purlin_status purlin_debug_drop_notify(purlin_handle h, long long item) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  std::lock_guard<std::mutex> lock(h->mu);
  h->drop_notify = item < 0 ? -1 : item;
  return PL_OK;
}

purlin_status purlin_debug_set_epoch(purlin_handle h, uint32_t epoch, purlin_stream_t stream) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  // the counter holds the epoch the last launch used, 0 .. 0xFFFFFFFE: from
  // 0xFFFFFFFF the next launch would take epoch 0, the value of cleared flags
  if (epoch == 0xFFFFFFFFu) return PL_ERR_INVALID_ARG;
  if (capturing((cudaStream_t)stream)) return PL_ERR_INVALID_ARG;  // a captured copy would read a dead stack slot
  std::lock_guard<std::mutex> lock(h->mu);
  cudaError_t e = cudaMemcpyAsync(h->ctl + pl::kCtlEpoch, &epoch, sizeof epoch, cudaMemcpyHostToDevice,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);  // `epoch` is on this stack
  return cuda_fail(e);
}

purlin_status purlin_debug_limit_buffer(purlin_handle h, int is_output, int rank, uint64_t bytes) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  if (rank < 0 || rank >= PURLIN_MAX_WORLD) return PL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(h->mu);
  h->limit_side = is_output ? 1 : 0;
  h->limit_rank = rank;
  h->limit_bytes = bytes;
  return PL_OK;
}

purlin_status purlin_trace_enable(purlin_handle h, void* buffer, size_t buffer_bytes) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  std::lock_guard<std::mutex> lock(h->mu);
  if (!buffer) {
    h->trace = nullptr;
    h->trace_cap = 0;
    return PL_OK;
  }
  if (((uintptr_t)buffer & 7u) || buffer_bytes < 8 + sizeof(pl::TraceRecord)) return PL_ERR_INVALID_ARG;
  const size_t cap = (buffer_bytes - 8) / sizeof(pl::TraceRecord);
  h->trace = (unsigned long long*)buffer;
  h->trace_cap = (uint32_t)std::min<size_t>(cap, 0xFFFFFFFFu);
  return PL_OK;
}

purlin_status purlin_workspace_query(purlin_handle h, size_t* bytes, int* grown) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  std::lock_guard<std::mutex> lock(h->mu);
  if (bytes) *bytes = h->ws_bytes;
  if (grown) *grown = h->ws_grown;
  return PL_OK;
}

purlin_status purlin_query(purlin_handle h, int* sm_count, int* arch, int* max_ctas_per_sm) {
  purlin_status st;
  if ((st = check_handle(h))) return st;
  if (sm_count) *sm_count = h->sm_count;
  if (arch) *arch = h->arch;
  if (max_ctas_per_sm) *max_ctas_per_sm = h->max_ctas_per_sm;
  return PL_OK;
}

purlin_status purlin_plan_describe(purlin_coll coll, int world, purlin_dtype dtype, const size_t* sizes,
                                   const uint64_t* src_addr, const uint64_t* dst_addr, int sm_count,
                                   const purlin_tune* tune, purlin_item* items, size_t cap, size_t* n_items,
                                   int* grid, int* n_flags) {
  if (!sizes || world < 1 || world > PURLIN_MAX_WORLD) return PL_ERR_INVALID_ARG;
  const size_t n = pl::n_sizes((int)coll, world);
  std::vector<uint64_t> sz(n);
  for (size_t i = 0; i < n; ++i) sz[i] = sizes[i];
  uint8_t sres[pl::kMaxWorld] = {}, dres[pl::kMaxWorld] = {};
  for (int r = 0; r < world; ++r) {
    if (src_addr) sres[r] = (uint8_t)(src_addr[r] & 15u);
    if (dst_addr) dres[r] = (uint8_t)(dst_addr[r] & 15u);
  }
  pl::Tune over;
  if (tune) std::memcpy(&over, tune, sizeof over);
  pl::Plan p;
  int st = pl::build_plan((int)coll, world, (int)dtype, sz.data(), n, sres, dres, sm_count, 0, over, &p);
  if (st) return (purlin_status)st;
  if (!pl::check_plan(p).empty()) return PL_ERR_INVALID_ARG;
  if (n_items) *n_items = p.items.size();
  if (grid) *grid = p.grid;
  if (n_flags) *n_flags = p.n_flags;
  if (items) {
    for (size_t i = 0; i < p.items.size() && i < cap; ++i) {
      const pl::Item& it = p.items[i];
      purlin_item& o = items[i];
      o.src_off = it.src_off;
      o.dst_off = it.dst_off;
      o.len = it.len;
      o.src_mask = it.src_mask;
      o.dst_mask = it.dst_mask;
      o.wait = it.wait;
      o.notify = it.notify;
      if (p.queue) {
        o.cta = 0xFFFFFFFFu;  // whichever CTA takes it from the queue
        o.order = (uint32_t)i;
      } else if (p.strided) {
        o.cta = (uint32_t)(i % (size_t)p.grid);
        o.order = (uint32_t)(i / (size_t)p.grid);
      } else {
        const auto up = std::upper_bound(p.cta_begin.begin(), p.cta_begin.end(), (uint32_t)i);
        const uint32_t c = (uint32_t)(up - p.cta_begin.begin()) - 1;
        o.cta = c;
        o.order = (uint32_t)i - p.cta_begin[c];
      }
    }
  }
  return PL_OK;
}

}  // extern "C"
