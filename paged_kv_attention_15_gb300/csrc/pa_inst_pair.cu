// Instances of the split kernel with paired consumer roles (pa_pair.cuh).
#include "pa_launch.h"
#include "pa_pair.cuh"

namespace pa {

template <int D, int MT, int KV, int TSL>
static SplitKernel pair_entry() {
  using C = PCfg<D, MT, KV == kKvFp8, TSL>;
  return SplitKernel{reinterpret_cast<const void*>(&pa_pair_kernel<D, MT, KV, TSL>), C::SMEM_FIXED, C::NS,
                     C::THREADS, kPairLaunchRegs, 0};
}

template <int D, int KV>
static SplitKernel pair_by_tiles(int row_tiles, int slice) {
  if (row_tiles == 1 && slice == 16) return pair_entry<D, 1, KV, 16>();
  if (row_tiles == 2 && slice == 16) return pair_entry<D, 2, KV, 16>();
  if (row_tiles == 2 && slice == 32) return pair_entry<D, 2, KV, 32>();
  return SplitKernel{nullptr, 0, 0, 0};
}

SplitKernel pair_kernel_fp8(int head_dim, int row_tiles, int slice) {
  if (head_dim == 128) return pair_by_tiles<128, kKvFp8>(row_tiles, slice);
  if (head_dim == 256) return pair_by_tiles<256, kKvFp8>(row_tiles, slice);
  return SplitKernel{nullptr, 0, 0, 0};
}

// 16-bit caches: the draft-block geometry, four row tiles (64 query rows per
// unit), every pair taking the whole stage (32 or 64 tokens).
SplitKernel pair_kernel_16(int head_dim, bool f16, int row_tiles, int slice) {
  if (head_dim != 128 || row_tiles != 4) return SplitKernel{nullptr, 0, 0, 0};
  if (slice == 32) return f16 ? pair_entry<128, 4, kKvF16, 32>() : pair_entry<128, 4, kKvBf16, 32>();
  if (slice == 64) return f16 ? pair_entry<128, 4, kKvF16, 64>() : pair_entry<128, 4, kKvBf16, 64>();
  return SplitKernel{nullptr, 0, 0, 0};
}

}  // namespace pa
