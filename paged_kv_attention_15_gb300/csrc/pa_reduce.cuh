// Split-K combine kernels (included by the C-ABI unit only); the row
// combine itself is `combine_row` in pa_kernels.cuh. Source: the MSLK pull request "[ROCm] Add FlyDSL
// paged-attention decode backend (dense + fp8) with benchmark" (Kernels:
// pa_decode_reduce, the split-K partial combine).
#pragma once

#include "pa_kernels.cuh"

namespace pa {

// Explicit splits: grid covers B*T*Hq rows, 4 rows (warps) per CTA.
__global__ void __launch_bounds__(128) pa_reduce_splits_kernel(const __grid_constant__ ReduceParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * 4 + warp;
  const size_t rows = (size_t)p.B * p.T * p.Hq;
  if (row >= rows) return;
  const size_t base = row * p.num_splits;
  wait_prerequisite_grids();  // the partials come from the split kernel
  const float* po = p.part_o + base * p.D;
  const float* pl = p.part_lse + base;
  const int D = p.D;
  combine_row(
      p.num_splits, D, [&](int k) { return po + (size_t)k * D; }, [&](int k) { return __ldcg(pl + k); },
      p.out + row * D, p.lse ? p.lse + row : nullptr, lane, p.out_f16 != 0);
}

// Balanced launch: grid (units, ceil(M / 4)); warp w of CTA (u, y) combines
// row 4y + w of unit u = b * NHG + hg from the pieces that the split CTAs
// i0..i1 covering the unit wrote to slots u + i. Units wholly inside one
// CTA's share, and sequences with no keys, were written by the split kernel.
__global__ void __launch_bounds__(128) pa_reduce_balanced_kernel(const __grid_constant__ ReduceParams p) {
  __shared__ long long s_sum[2][4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  const int b = u / p.NHG, hg = u % p.NHG;
  const int cap = p.max_blocks * p.P;
  long long before = 0, total = 0;
  for (int i = threadIdx.x; i < p.B; i += 128) {
    int c = __ldg(p.context_lens + i);
    c = c < 0 ? 0 : (c > cap ? cap : c);
    const long long nv = (c + p.P - 1) / p.P + p.tidar;
    total += nv;
    if (i < b) before += nv;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if (lane == 0) {
    s_sum[0][warp] = before;
    s_sum[1][warp] = total;
  }
  __syncthreads();
  const int rho = blockIdx.y * 4 + warp;
  if (rho >= p.M) return;
  before = s_sum[0][0] + s_sum[0][1] + s_sum[0][2] + s_sum[0][3];
  total = s_sum[1][0] + s_sum[1][1] + s_sum[1][2] + s_sum[1][3];
  int cb = __ldg(p.context_lens + b);
  cb = cb < 0 ? 0 : (cb > cap ? cap : cb);
  const long long nvb = (cb + p.P - 1) / p.P + p.tidar;
  if (nvb == 0) return;
  const long long N = total * p.NHG;
  const long long us = before * p.NHG + (long long)hg * nvb;
  const long long ue = us + nvb;
  const long long G64 = p.grid;
  const int i0 = (int)(((us + 1) * G64 - 1) / N);
  const int i1 = (int)((ue * G64 - 1) / N);
  if (i0 == i1) return;  // one piece: the split kernel wrote the final rows
  // row rho = hl * GT + t * G + j -> query head (hg * H2 + hl) * G + j
  const int hl = rho / p.GT, rem = rho - hl * p.GT;
  const int t = rem / p.G;
  const size_t row = ((size_t)b * p.T + t) * p.Hq + (size_t)(hg * p.H2 + hl) * p.G + (rem - t * p.G);
  wait_prerequisite_grids();  // the partials come from the split kernel
  const float* po = p.part_o;
  const float* pl = p.part_lse;
  const int M = p.M, D = p.D;
  const float NEG_INF = -__int_as_float(0x7f800000);
  combine_row(
      i1 - i0 + 1, D, [&](int k) { return po + ((size_t)(u + i0 + k) * M + rho) * D; },
      [&](int k) {
        const long long i = i0 + k;  // a CTA whose share is empty wrote nothing
        return (N * i / G64) < (N * (i + 1) / G64) ? __ldcg(pl + (size_t)(u + i) * M + rho) : NEG_INF;
      },
      p.out + row * D, p.lse ? p.lse + row : nullptr, lane, p.out_f16 != 0);
}

}  // namespace pa
