// 16-bit KV instances of the split kernel: bf16, or f16 when this file is
// included by pa_inst_f16.cu with PA_INST_KV / PA_INST_FN set.
#include "pa_launch.h"

namespace pa {

#ifndef PA_INST_KV
#define PA_INST_KV kKvBf16
#define PA_INST_FN split_kernel_bf16
#endif
constexpr int KVK = PA_INST_KV;

template <int D, int MT, int TSL, int CW = kConsumerWarps>
static SplitKernel entry() {
  using C = Cfg<D, MT, false, TSL, CW>;
  return SplitKernel{reinterpret_cast<const void*>(&pa_split_kernel<D, MT, KVK, TSL, CW>), C::SMEM_FIXED, C::NS,
                     C::THREADS, C::REGSPLIT ? kSplitLaunchRegs : 0, C::FUSED ? 1 : 0};
}

template <int D>
static SplitKernel by_tiles(int row_tiles, int slice, int cw) {
  if constexpr (D == 128) {
    // eight consumer warps, two per row tile: the four-tile draft-block
    // units (64 query rows of one or two kv heads), in 16-token slices or
    // (with the register split) 32-token slices
    if (cw == 8) {
      if (row_tiles == 4 && slice == 16) return entry<D, 4, 16, 8>();
      if (row_tiles == 4 && slice == 32) return entry<D, 4, 32, 8>();
      return SplitKernel{nullptr, 0, 0, 0};
    }
  }
  if constexpr (D == 64) {
    // eight consumer warps, four per row tile, one kv head each: GQA units
    // of eight kv heads (G T = 4), whose page box of 16 rows x 8 heads x
    // 128 B is 16 KB
    if (cw == 8) {
      if (row_tiles == 2 && slice == 16) return entry<D, 2, 16, 8>();
      return SplitKernel{nullptr, 0, 0, 0};
    }
  }
  if (cw != kConsumerWarps) return SplitKernel{nullptr, 0, 0, 0};
  if (row_tiles == 1 && slice == 16) return entry<D, 1, 16>();
  if constexpr (D == 64) {  // 128-row stages: 32 tokens per warp with one row tile
    if (row_tiles == 1 && slice == 32) return entry<D, 1, 32>();
  }
  if (row_tiles == 2 && slice == 16) return entry<D, 2, 16>();
  if (row_tiles == 2 && slice == 32) return entry<D, 2, 32>();
  if constexpr (D == 128 || D == 64) {
    // four row tiles: up to 64 query rows (long draft blocks); a slice of
    // 64 tokens when one kv head fills the tiles
    if (row_tiles == 4 && slice == 16) return entry<D, 4, 16>();
    if (row_tiles == 4 && slice == 32) return entry<D, 4, 32>();
    if (row_tiles == 4 && slice == 64) return entry<D, 4, 64>();
  }
  return SplitKernel{nullptr, 0, 0, 0};
}

SplitKernel PA_INST_FN(int head_dim, int row_tiles, int slice, int cw) {
  if (head_dim == 64) return by_tiles<64>(row_tiles, slice, cw);
  if (head_dim == 128) return by_tiles<128>(row_tiles, slice, cw);
  if (head_dim == 256) return by_tiles<256>(row_tiles, slice, cw);
  return SplitKernel{nullptr, 0, 0, 0};
}

}  // namespace pa
