// Copy-only kernels: AllGather(V), AllToAll(V) and the copy Atom entry point.
#include "kernels.cuh"

namespace pl {

const void* kernel_copy(int unroll) {
  switch (unroll) {
    case 1: return (const void*)snac_kernel<void, 1, 1>;
    case 2: return (const void*)snac_kernel<void, 1, 2>;
    case 4: return (const void*)snac_kernel<void, 1, 4>;
    case 8: return (const void*)snac_kernel<void, 1, 8>;
    default: return nullptr;
  }
}

}  // namespace pl
