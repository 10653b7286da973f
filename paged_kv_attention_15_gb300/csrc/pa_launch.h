// Internal interface between the C-ABI host code and the kernel instances.
#pragma once

#include <cuda_runtime.h>

#include "pa_kernels.cuh"

namespace pa {

struct SplitKernel {
  const void* fn;   // __global__ function, launched with cudaLaunchKernel
  int smem_fixed;   // dynamic shared memory without the per-sequence table
  int stages;       // pipeline depth of the instance
  int threads;      // block size: 32 * (consumer warps + 1), or whole warpgroups
  int launch_regs;  // kernels that move registers between warpgroups (setmaxnreg):
                    // the registers per thread their split needs at launch; 0 otherwise
  int fused;        // 1: the balanced schedule's combine can be fused into this kernel
};

// Kernel instance for (head_dim, row tiles, tokens per warp slice,
// consumer warps); fn == nullptr if that combination is not built.
SplitKernel split_kernel_bf16(int head_dim, int row_tiles, int slice, int consumer_warps);
SplitKernel split_kernel_fp8(int head_dim, int row_tiles, int slice, int consumer_warps);
SplitKernel split_kernel_f16(int head_dim, int row_tiles, int slice, int consumer_warps);

// Instance of the split kernel with paired consumer roles (per row tile and
// slice group an S warp and two PV warps, four such pairs) for (head_dim,
// row tiles, tokens per warp slice); fn == nullptr if not built.
SplitKernel pair_kernel_fp8(int head_dim, int row_tiles, int slice);
SplitKernel pair_kernel_16(int head_dim, bool f16, int row_tiles, int slice);

// Instance of the tcgen05 kernel for (head_dim, query rows per kv head GT,
// rows per work unit N = kv heads per unit * GT); fn == nullptr if not built.
SplitKernel umma_kernel_fp8(int head_dim, int GT, int N);
SplitKernel umma_kernel_16(int head_dim, bool f16, int GT, int N);

// Instance of the query-row-major tcgen05 kernel (16-bit caches) for
// (head_dim, kv heads per unit, query rows per unit m = 64 or 128);
// fn == nullptr if not built.
SplitKernel qrow_kernel_16(int head_dim, bool f16, int h2, int m);

}  // namespace pa
