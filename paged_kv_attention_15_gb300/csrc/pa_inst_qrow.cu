// Instances of the query-row-major tcgen05 kernel: bf16 and f16 caches,
// D = 128, units of two kv heads x 32 query rows or one kv head x 64 (64
// rows), or four kv heads x 32 (128 rows).
#include "pa_launch.h"
#include "pa_qrow.cuh"

namespace pa {

template <int D, int KV, int H2, int M>
static SplitKernel qentry() {
  using C = QCfg<D, M>;
  return SplitKernel{reinterpret_cast<const void*>(&pa_qrow_kernel<D, KV, H2, M>), C::SMEM_FIXED, C::NS, kQThreads,
                     0};
}

SplitKernel qrow_kernel_16(int head_dim, bool f16, int h2, int m) {
  if (head_dim != 128) return SplitKernel{nullptr, 0, 0, 0, 0};
  if (m == 64 && h2 == 1) return f16 ? qentry<128, kKvF16, 1, 64>() : qentry<128, kKvBf16, 1, 64>();
  if (m == 64 && h2 == 2) return f16 ? qentry<128, kKvF16, 2, 64>() : qentry<128, kKvBf16, 2, 64>();
  if (m == 128 && h2 == 4) return f16 ? qentry<128, kKvF16, 4, 128>() : qentry<128, kKvBf16, 4, 128>();
  return SplitKernel{nullptr, 0, 0, 0, 0};
}

}  // namespace pa
