// TMA bulk pipeline kernels: copies (AllGather(V), AllToAll(V), copy Atom)
// and reductions over fp32 / bf16 with 2..8 sources (plus a generic count).
#include "kernels_bulk.cuh"

namespace pl {

const void* kernel_bulk_copy() { return (const void*)bulk_kernel<void, 1>; }

template <typename T>
static const void* pick_bulk_reduce(int nsrc) {
  switch (nsrc) {
    case 2: return (const void*)bulk_kernel<T, 2>;
    case 3: return (const void*)bulk_kernel<T, 3>;
    case 4: return (const void*)bulk_kernel<T, 4>;
    case 5: return (const void*)bulk_kernel<T, 5>;
    case 6: return (const void*)bulk_kernel<T, 6>;
    case 7: return (const void*)bulk_kernel<T, 7>;
    case 8: return (const void*)bulk_kernel<T, 8>;
    default: return (nsrc >= 2 && nsrc <= kMaxWorld) ? (const void*)bulk_kernel<T, 0> : nullptr;
  }
}

const void* kernel_bulk_reduce_f32(int nsrc) { return pick_bulk_reduce<float>(nsrc); }
const void* kernel_bulk_reduce_bf16(int nsrc) { return pick_bulk_reduce<bf16_tag>(nsrc); }

}  // namespace pl
