// bf16 KV instances of the split kernel.
#include "pa_launch.h"

namespace pa {

template <int D, int MT>
static SplitKernel entry() {
  using C = Cfg<D, MT, false>;
  return SplitKernel{reinterpret_cast<const void*>(&pa_split_kernel<D, MT, false>), C::SMEM_FIXED, C::NS};
}

SplitKernel split_kernel_bf16(int head_dim, int row_tiles) {
  if (row_tiles == 1) {
    if (head_dim == 64) return entry<64, 1>();
    if (head_dim == 128) return entry<128, 1>();
    if (head_dim == 256) return entry<256, 1>();
  } else if (row_tiles == 2) {
    if (head_dim == 64) return entry<64, 2>();
    if (head_dim == 128) return entry<128, 2>();
    if (head_dim == 256) return entry<256, 2>();
  }
  return SplitKernel{nullptr, 0, 0};
}

}  // namespace pa
