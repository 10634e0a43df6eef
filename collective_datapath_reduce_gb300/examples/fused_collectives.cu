// Example: a user kernel that fuses its own work with a device-side collective
// (purlin 0.6.5, "Device-side": do some work, call the collective, do some
// other work), built on include/purlin_device.cuh only.
//
// Work before the call (optional): every CTA writes part of the ranks' source
// buffers (byte transform x ^ 0x5A for the copy collectives, a plain copy for
// the reductions), so the collective must see other CTAs' writes.  Work after
// (optional): every CTA reads part of the destinations and writes
// dst + 1 (per byte) to `post`, so the call must have finished everywhere.
// Built into libpurlin_examples.so; the tests check it against the CPU oracle
// and the benchmark times the bare device-side collective with it.
#include <cuda_runtime.h>

#include "purlin_device.cuh"

namespace {

struct FusedArgs {
  purlin::Context ctx;
  const unsigned char* in[purlin::kMaxRanks];  // inputs of the work before the call
  unsigned char* post[purlin::kMaxRanks];      // results of the work after the call
  unsigned long long bytes;                    // per-rank input bytes
  unsigned long long out_bytes;                // per-rank output bytes
  int which;                                   // 0 AG, 1 A2A, 2 AR bf16, 3 RS fp32, 4 AR fp32 world 8;
                                               // 5 AG and 6 AR bf16 with evict-first stores,
                                               // 7 AR bf16 with one vector per source in flight
  int coll_blocks;
  int* status;
  int work;                                    // bit 0: work before the call, bit 1: work after
};

__global__ void __launch_bounds__(256) fused_kernel(const __grid_constant__ FusedArgs f) {
  const int N = f.ctx.world;
  const unsigned long long tid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  const unsigned long long nth = (unsigned long long)gridDim.x * blockDim.x;
  if (f.work & 1) {
    const unsigned long long total = (unsigned long long)N * f.bytes;
    for (unsigned long long k = tid; k < total; k += nth) {
      const int r = (int)(k / f.bytes);
      const unsigned long long i = k % f.bytes;
      const unsigned char x = f.in[r][i];
      const bool copy = f.which <= 1 || f.which == 5;
      const_cast<char*>(f.ctx.src[r])[i] = (char)(copy ? (x ^ 0x5A) : x);
    }
  }
  const purlin::SnacArgs a{f.bytes, (int)gridDim.x, f.coll_blocks, (int)blockIdx.x, (f.work & 2) != 0};
  int st;
  switch (f.which) {
    case 0: st = purlin::all_gather(a, f.ctx); break;
    case 1: st = purlin::all_to_all(a, f.ctx); break;
    case 2:  // the source count as a template argument when it is the common 8
      st = N == 8 ? purlin::all_reduce<pl::bf16_tag, 8>(a, f.ctx) : purlin::all_reduce<pl::bf16_tag>(a, f.ctx);
      break;
    case 3: st = purlin::reduce_scatter<float>(a, f.ctx); break;
    case 5: st = purlin::all_gather<true>(a, f.ctx); break;
    case 6:
      st = N == 8 ? purlin::all_reduce<pl::bf16_tag, 8, 2, true>(a, f.ctx)
                  : purlin::all_reduce<pl::bf16_tag, 0, 2, true>(a, f.ctx);
      break;
    case 7:  // one vector per source in flight (the smallest register footprint)
      st = N == 8 ? purlin::all_reduce<pl::bf16_tag, 8, 1>(a, f.ctx) : purlin::all_reduce<pl::bf16_tag, 0, 1>(a, f.ctx);
      break;
    default: st = purlin::all_reduce<float, 8>(a, f.ctx); break;
  }
  if (threadIdx.x == 0 && st != purlin::kOk) atomicExch(f.status, st);
  if (f.work & 2) {
    const unsigned long long otot = (unsigned long long)N * f.out_bytes;
    for (unsigned long long k = tid; k < otot; k += nth) {
      const int r = (int)(k / f.out_bytes);
      const unsigned long long i = k % f.out_bytes;
      f.post[r][i] = (unsigned char)(__ldcg(reinterpret_cast<const unsigned char*>(f.ctx.dst[r]) + i) + 1);
    }
  }
}

}  // namespace

extern "C" int purlin_example_fused_args_bytes() { return (int)sizeof(FusedArgs); }

// Largest grid whose CTAs are all resident (every CTA enters the collective).
extern "C" int purlin_example_fused_max_grid(int* grid) {
  int dev = 0, sms = 0, occ = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 2;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fused_kernel, 256, 0) != cudaSuccess) return 3;
  *grid = occ * sms;
  return 0;
}

// Cooperative launch: every CTA that enters the collective is resident.
extern "C" int purlin_example_fused_launch(const void* args, int grid, void* stream) {
  FusedArgs f = *static_cast<const FusedArgs*>(args);
  void* kargs[] = {&f};
  const cudaError_t e = cudaLaunchCooperativeKernel((const void*)fused_kernel, dim3(grid), dim3(256), kargs, 0,
                                                    (cudaStream_t)stream);
  return e == cudaSuccess ? 0 : (int)e;
}
