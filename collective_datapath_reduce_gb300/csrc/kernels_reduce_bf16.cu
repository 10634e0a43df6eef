// Reduce kernels over bf16 data: AllReduce (both layouts), ReduceScatter(V)
// and the reduce Atom entry point.  One variant per source count up to 8
// (all loads of a vector issued before the first add) and one for any count
// up to 16 (loads in batches of 8).
#include "kernels.cuh"

namespace pl {

const void* kernel_reduce_bf16(int nsrc, int unroll) {
  const bool u2 = unroll >= 2;
  switch (nsrc) {
    case 2: return u2 ? (const void*)snac_kernel<bf16_tag, 2, 2> : (const void*)snac_kernel<bf16_tag, 2, 1>;
    case 3: return u2 ? (const void*)snac_kernel<bf16_tag, 3, 2> : (const void*)snac_kernel<bf16_tag, 3, 1>;
    case 4: return u2 ? (const void*)snac_kernel<bf16_tag, 4, 2> : (const void*)snac_kernel<bf16_tag, 4, 1>;
    case 5: return (const void*)snac_kernel<bf16_tag, 5, 1>;
    case 6: return (const void*)snac_kernel<bf16_tag, 6, 1>;
    case 7: return (const void*)snac_kernel<bf16_tag, 7, 1>;
    case 8: return (const void*)snac_kernel<bf16_tag, 8, 1>;
    default: return (nsrc >= 2 && nsrc <= kMaxWorld) ? (const void*)snac_kernel<bf16_tag, 0, 1> : nullptr;
  }
}

// Ring AllReduce: each reduce stage adds one rank's input to the running
// binary32 sum another CTA stored, as two 16-bit halves, earlier in this
// launch (loads through the L2).
const void* kernel_reduce_ring_bf16(int unroll) {
  return unroll >= 2 ? (const void*)snac_kernel<bf16_tag, 2, 2, kKindRing> : (const void*)snac_kernel<bf16_tag, 2, 1, kKindRing>;
}

}  // namespace pl
