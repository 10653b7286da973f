// fp8 (e4m3fn) KV instances of the split kernel.
#include "pa_launch.h"

namespace pa {

template <int D, int MT, int TSL, int CW = kConsumerWarps>
static SplitKernel entry() {
  using C = Cfg<D, MT, true, TSL, CW>;
  return SplitKernel{reinterpret_cast<const void*>(&pa_split_kernel<D, MT, kKvFp8, TSL, CW>), C::SMEM_FIXED, C::NS,
                     C::THREADS, C::REGSPLIT ? kSplitLaunchRegs : 0, C::FUSED ? 1 : 0};
}

template <int D>
static SplitKernel by_tiles(int row_tiles, int slice, int cw) {
  if (cw != kConsumerWarps) return SplitKernel{nullptr, 0, 0, 0};
  if (row_tiles == 1 && slice == 16) return entry<D, 1, 16>();
  if (row_tiles == 2 && slice == 16) return entry<D, 2, 16>();
  if (row_tiles == 2 && slice == 32) return entry<D, 2, 32>();
  return SplitKernel{nullptr, 0, 0, 0};
}

SplitKernel split_kernel_fp8(int head_dim, int row_tiles, int slice, int cw) {
  if (head_dim == 128) return by_tiles<128>(row_tiles, slice, cw);
  if (head_dim == 256) return by_tiles<256>(row_tiles, slice, cw);
  return SplitKernel{nullptr, 0, 0, 0};
}

}  // namespace pa
