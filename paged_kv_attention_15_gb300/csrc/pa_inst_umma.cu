// Instances of the tcgen05 decode kernel: 16-bit caches (bf16 and f16,
// D = 128) when this file is compiled alone; fp8 caches (D = 128, 256) when
// included by pa_inst_umma_fp8.cu with PA_UMMA_FP8 set.
#include "pa_launch.h"
#include "pa_umma.cuh"

namespace pa {

template <int D, int KV, int GT, int N>
static SplitKernel uentry() {
  using C = UCfg<D, KV, GT, N>;
  if constexpr (C::FITS) {
    return SplitKernel{reinterpret_cast<const void*>(&pa_umma_kernel<D, KV, GT, N>), C::SMEM_FIXED, C::NRAW,
                       kUThreads, kULaunchRegs};
  } else {
    return SplitKernel{nullptr, 0, 0, 0};
  }
}

// (query rows per kv head, rows per unit) pairs built for every format.
template <int D, int KV>
static SplitKernel by_rows(int GT, int N) {
  if (GT == 16 && N == 16) return uentry<D, KV, 16, 16>();
  if (GT == 16 && N == 32) return uentry<D, KV, 16, 32>();
  if (GT == 16 && N == 64) return uentry<D, KV, 16, 64>();
  if (GT == 32 && N == 32) return uentry<D, KV, 32, 32>();
  if (GT == 32 && N == 64) return uentry<D, KV, 32, 64>();
  return SplitKernel{nullptr, 0, 0, 0};
}

#ifdef PA_UMMA_FP8
SplitKernel umma_kernel_fp8(int head_dim, int GT, int N) {
  if (head_dim == 128) return by_rows<128, kKvFp8>(GT, N);
  if (head_dim == 256) return by_rows<256, kKvFp8>(GT, N);
  return SplitKernel{nullptr, 0, 0, 0};
}
#else
SplitKernel umma_kernel_16(int head_dim, bool f16, int GT, int N) {
  if (head_dim != 128) return SplitKernel{nullptr, 0, 0, 0};
  return f16 ? by_rows<128, kKvF16>(GT, N) : by_rows<128, kKvBf16>(GT, N);
}
#endif

}  // namespace pa
