// Reduce kernels of two-shot AllReduce plans with L2 priorities (store_hint
// 3): reduce inputs loaded evict-first, owner tiles stored evict-last until
// their copies read them, copies stored evict-first.  The same variants per
// source count as the plain reduce kernels, for both element types.
#include "kernels.cuh"

namespace pl {

namespace {

template <typename T>
const void* l2_kernel(int nsrc, int unroll) {
  const bool u2 = unroll >= 2;
  switch (nsrc) {
    case 2: return u2 ? (const void*)snac_kernel<T, 2, 2, kKindL2> : (const void*)snac_kernel<T, 2, 1, kKindL2>;
    case 3: return u2 ? (const void*)snac_kernel<T, 3, 2, kKindL2> : (const void*)snac_kernel<T, 3, 1, kKindL2>;
    case 4: return u2 ? (const void*)snac_kernel<T, 4, 2, kKindL2> : (const void*)snac_kernel<T, 4, 1, kKindL2>;
    case 5: return (const void*)snac_kernel<T, 5, 1, kKindL2>;
    case 6: return (const void*)snac_kernel<T, 6, 1, kKindL2>;
    case 7: return (const void*)snac_kernel<T, 7, 1, kKindL2>;
    case 8: return (const void*)snac_kernel<T, 8, 1, kKindL2>;
    default: return (nsrc >= 2 && nsrc <= kMaxWorld) ? (const void*)snac_kernel<T, 0, 1, kKindL2> : nullptr;
  }
}

}  // namespace

const void* kernel_reduce_l2_f32(int nsrc, int unroll) { return l2_kernel<float>(nsrc, unroll); }
const void* kernel_reduce_l2_bf16(int nsrc, int unroll) { return l2_kernel<bf16_tag>(nsrc, unroll); }

}  // namespace pl
