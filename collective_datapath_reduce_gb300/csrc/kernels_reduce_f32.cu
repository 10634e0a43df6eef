// Reduce kernels over f32 data: AllReduce (both layouts), ReduceScatter(V)
// and the reduce Atom entry point.  One variant per source count up to 8
// (all loads of a vector issued before the first add) and one for any count
// up to 16 (loads in batches of 8).
#include "kernels.cuh"

namespace pl {

const void* kernel_reduce_f32(int nsrc, int unroll) {
  const bool u2 = unroll >= 2;
  switch (nsrc) {
    case 2: return u2 ? (const void*)snac_kernel<float, 2, 2> : (const void*)snac_kernel<float, 2, 1>;
    case 3: return u2 ? (const void*)snac_kernel<float, 3, 2> : (const void*)snac_kernel<float, 3, 1>;
    case 4: return u2 ? (const void*)snac_kernel<float, 4, 2> : (const void*)snac_kernel<float, 4, 1>;
    case 5: return (const void*)snac_kernel<float, 5, 1>;
    case 6: return (const void*)snac_kernel<float, 6, 1>;
    case 7: return (const void*)snac_kernel<float, 7, 1>;
    case 8: return (const void*)snac_kernel<float, 8, 1>;
    default: return (nsrc >= 2 && nsrc <= kMaxWorld) ? (const void*)snac_kernel<float, 0, 1> : nullptr;
  }
}

// Ring AllReduce: each reduce stage adds one rank's input to the running sum
// another CTA stored earlier in this launch (loads through the L2).
const void* kernel_reduce_ring_f32(int unroll) {
  return unroll >= 2 ? (const void*)snac_kernel<float, 2, 2, kKindRing> : (const void*)snac_kernel<float, 2, 1, kKindRing>;
}

}  // namespace pl
