// Split-K combine kernels (included by the C-ABI unit only).
//
// One warp per query row: M = max_k lse_k, w_k = exp(lse_k - M),
// out = sum_k w_k o_k / sum_k w_k, lse = M + ln sum_k w_k; pieces with
// lse = -inf weigh 0 and a row whose pieces are all empty gets out = 0,
// lse = -inf. Source: the MSLK pull request "[ROCm] Add FlyDSL
// paged-attention decode backend (dense + fp8) with benchmark" (Kernels:
// pa_decode_reduce, the split-K partial combine).
#pragma once

#include "pa_kernels.cuh"

namespace pa {

// Combines the pieces k = 0..np-1 of one row; piece k's partial is the D
// floats at o_row(k) and its lse is at *l_row(k). Lane l holds the lse and
// weight of pieces l, l+32, ...; weights are broadcast by shuffle so the
// partial loads of a warp are independent of one another.
template <typename ORow, typename LRow>
__device__ __forceinline__ void combine_row(int np, int D, ORow o_row, LRow l_row, __nv_bfloat16* out,
                                            float* lse_out, int lane) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float LOG2E = 1.4426950408889634f;
  float mx = NEG_INF;
  for (int k = lane; k < np; k += 32) mx = fmaxf(mx, *l_row(k));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (mx == NEG_INF) {
    for (int d = lane * 4; d < D; d += 128) *reinterpret_cast<uint2*>(out + d) = make_uint2(0u, 0u);
    if (lane == 0 && lse_out) *lse_out = NEG_INF;
    return;
  }
  float L = 0.f;
  for (int k = lane; k < np; k += 32) {
    const float lk = *l_row(k);
    L += lk == NEG_INF ? 0.f : ex2((lk - mx) * LOG2E);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = 1.f / L;
  for (int d0 = 0; d0 < D; d0 += 128) {  // one float4 per lane per pass
    const int dd = d0 + lane * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < np; k0 += 32) {
      const float lk = k0 + lane < np ? *l_row(k0 + lane) : NEG_INF;
      const float wk = lk == NEG_INF ? 0.f : ex2((lk - mx) * LOG2E);
      const int n = np - k0 < 32 ? np - k0 : 32;
#pragma unroll 4
      for (int i = 0; i < n; ++i) {
        const float w = __shfl_sync(0xffffffffu, wk, i);
        if (dd < D && w != 0.f) {
          const float4 v = *reinterpret_cast<const float4*>(o_row(k0 + i) + dd);
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
      }
    }
    if (dd < D)
      *reinterpret_cast<uint2*>(out + dd) =
          make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  }
  if (lane == 0 && lse_out) *lse_out = mx + lg2(L) * kLn2;
}

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
      p.num_splits, D, [&](int k) { return po + (size_t)k * D; }, [&](int k) { return pl + k; },
      p.out + row * D, p.lse ? p.lse + row : nullptr, lane);
}

// Output row of row rho of unit (b, hg) in [B, T, Hq]: query token
// t = (rho % GT) / G of head (hg * H2 + rho / GT) * G + rho % G.
__device__ __forceinline__ size_t unit_row(const ReduceParams& p, int b, int hg, int rho) {
  const int hl = rho / p.GT, rem = rho - hl * p.GT;
  const int t = rem / p.G;
  return ((size_t)b * p.T + t) * p.Hq + (size_t)(hg * p.H2 + hl) * p.G + (rem - t * p.G);
}

// Balanced launch: grid (units, ceil(M / 4)); warp w of CTA (u, y) combines
// row 4y + w of unit u = b * NHG + hg from the pieces that the split CTAs
// i0..i1 covering the unit wrote to slots u + i.
__global__ void __launch_bounds__(128) pa_reduce_balanced_kernel(const __grid_constant__ ReduceParams p) {
  __shared__ long long s_sum[2][4];
  __shared__ float s_ninf;  // lse of a piece whose CTA share was empty
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s_ninf = -__int_as_float(0x7f800000);
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
  const long long N = total * p.NHG;
  const long long us = before * p.NHG + (long long)hg * nvb;
  const long long ue = us + nvb;
  const size_t row = unit_row(p, b, hg, rho);
  const float NEG_INF = -__int_as_float(0x7f800000);
  if (nvb == 0) {  // no keys at all: out = 0, lse = -inf
    for (int d = lane * 4; d < p.D; d += 128) *reinterpret_cast<uint2*>(p.out + row * p.D + d) = make_uint2(0u, 0u);
    if (lane == 0 && p.lse) p.lse[row] = NEG_INF;
    return;
  }
  const long long G64 = p.grid;
  const int i0 = (int)(((us + 1) * G64 - 1) / N);
  const int i1 = (int)((ue * G64 - 1) / N);
  if (i0 == i1) return;  // one piece: the split kernel wrote the final rows
  wait_prerequisite_grids();  // the partials come from the split kernel
  // CTAs whose share is empty wrote nothing: their lse reads as -inf here.
  const float* po = p.part_o;
  const float* pl = p.part_lse;
  const int M = p.M, D = p.D;
  const float* empty_lse = &s_ninf;
  combine_row(
      i1 - i0 + 1, D,
      [&](int k) { return po + ((size_t)(u + i0 + k) * M + rho) * D; },
      [&](int k) -> const float* {
        const long long i = i0 + k;
        return (N * i / G64) < (N * (i + 1) / G64) ? pl + (size_t)(u + i) * M + rho : empty_lse;
      },
      p.out + row * D, p.lse ? p.lse + row : nullptr, lane);
}

}  // namespace pa
