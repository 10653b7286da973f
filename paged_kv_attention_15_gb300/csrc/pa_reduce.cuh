// Split-K combine kernels (included by the C-ABI unit only).
#pragma once

#include "pa_kernels.cuh"

namespace pa {

// ----------------------------------------------------------- reduce kernel
// One warp per query row: M = max_k lse_k, w_k = exp(lse_k - M),
// out = sum_k w_k o_k / sum_k w_k, lse = M + ln sum_k w_k.
__device__ __forceinline__ void reduce_row(const ReduceParams& p, size_t row, const float* po, const float* pl,
                                           size_t stride_piece, int npieces, int lane) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float LOG2E = 1.4426950408889634f;
  float mx = NEG_INF;
  for (int k = lane; k < npieces; k += 32) mx = fmaxf(mx, pl[k * stride_piece]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __nv_bfloat16* out = p.out + row * p.D;
  if (mx == NEG_INF) {
    for (int d = lane * 4; d < p.D; d += 128) {
      *reinterpret_cast<uint2*>(out + d) = make_uint2(0u, 0u);
    }
    if (lane == 0 && p.lse) p.lse[row] = NEG_INF;
    return;
  }
  float L = 0.f;
  for (int k = lane; k < npieces; k += 32) L += ex2((pl[k * stride_piece] - mx) * LOG2E);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = 1.f / L;
  for (int d = lane * 4; d < p.D; d += 128) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < npieces; ++k) {
      const float w = ex2((pl[k * stride_piece] - mx) * LOG2E);
      if (w == 0.f) continue;
      const float4 v = *reinterpret_cast<const float4*>(po + k * stride_piece * p.D + d);
      a.x += w * v.x;
      a.y += w * v.y;
      a.z += w * v.z;
      a.w += w * v.w;
    }
    *reinterpret_cast<uint2*>(out + d) = make_uint2(pack_bf16x2(a.x * inv, a.y * inv), pack_bf16x2(a.z * inv, a.w * inv));
  }
  if (lane == 0 && p.lse) p.lse[row] = (mx + lg2(L) * kLn2);
}

// Output row of row rho of unit (b, hg) in [B, T, Hq].
__device__ __forceinline__ size_t unit_row(const ReduceParams& p, int b, int hg, int rho) {
  const int hl = rho / p.GT, rem = rho - hl * p.GT;
  const int t = rem / p.G;
  return ((size_t)b * p.T + t) * p.Hq + (size_t)(hg * p.H2 + hl) * p.G + (rem - t * p.G);
}

// Explicit splits: grid covers B*T*Hq rows, 4 rows (warps) per CTA.
__global__ void __launch_bounds__(128) pa_reduce_splits_kernel(const __grid_constant__ ReduceParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * 4 + warp;
  const size_t rows = (size_t)p.B * p.T * p.Hq;
  if (row >= rows) return;
  const size_t base = row * p.num_splits;
  wait_prerequisite_grids();  // the partials come from the split kernel
  reduce_row(p, row, p.part_o + base * p.D, p.part_lse + base, 1, p.num_splits, lane);
}

// Balanced launch: one CTA per (sequence, head group) unit; combines the
// pieces that the split CTAs wrote to slots unit + cta. Row rho of a unit is
// query token t = (rho % GT) / G of head (hg * H2 + rho / GT) * G + rho % G.
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
  before = s_sum[0][0] + s_sum[0][1] + s_sum[0][2] + s_sum[0][3];
  total = s_sum[1][0] + s_sum[1][1] + s_sum[1][2] + s_sum[1][3];
  int cb = __ldg(p.context_lens + b);
  cb = cb < 0 ? 0 : (cb > cap ? cap : cb);
  const long long nvb = (cb + p.P - 1) / p.P + p.tidar;
  const long long N = total * p.NHG;
  const long long us = before * p.NHG + (long long)hg * nvb;
  const long long ue = us + nvb;
  const float NEG_INF = -__int_as_float(0x7f800000);
  if (nvb == 0) {  // no keys at all: out = 0, lse = -inf
    for (int rho = warp; rho < p.M; rho += 4) {
      const size_t row = unit_row(p, b, hg, rho);
      for (int d = lane * 4; d < p.D; d += 128) *reinterpret_cast<uint2*>(p.out + row * p.D + d) = make_uint2(0u, 0u);
      if (lane == 0 && p.lse) p.lse[row] = NEG_INF;
    }
    return;
  }
  wait_prerequisite_grids();  // the partials and final rows come from the split kernel
  const long long G64 = p.grid;
  const int i0 = (int)(((us + 1) * G64 - 1) / N);
  const int i1 = (int)((ue * G64 - 1) / N);
  if (i0 == i1) return;  // one piece: the split kernel wrote the final rows
  // Pieces are the CTAs i0..i1 whose share is non-empty; slot = u + i.
  for (int rho = warp; rho < p.M; rho += 4) {
    const size_t row = unit_row(p, b, hg, rho);
    float mx = NEG_INF;
    for (int i = i0 + lane; i <= i1; i += 32) {
      const bool nonempty = (N * i / G64) < (N * (i + 1) / G64);
      if (nonempty) mx = fmaxf(mx, p.part_lse[(size_t)(u + i) * p.M + rho]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __nv_bfloat16* out = p.out + row * p.D;
    if (mx == NEG_INF) {
      for (int d = lane * 4; d < p.D; d += 128) *reinterpret_cast<uint2*>(out + d) = make_uint2(0u, 0u);
      if (lane == 0 && p.lse) p.lse[row] = NEG_INF;
      continue;
    }
    const float LOG2E = 1.4426950408889634f;
    float L = 0.f;
    for (int i = i0 + lane; i <= i1; i += 32) {
      const bool nonempty = (N * i / G64) < (N * (i + 1) / G64);
      if (nonempty) L += ex2((p.part_lse[(size_t)(u + i) * p.M + rho] - mx) * LOG2E);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float inv = 1.f / L;
    for (int d = lane * 4; d < p.D; d += 128) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = i0; i <= i1; ++i) {
        if (!((N * i / G64) < (N * (i + 1) / G64))) continue;
        const size_t slot_row = (size_t)(u + i) * p.M + rho;
        const float w = ex2((p.part_lse[slot_row] - mx) * LOG2E);
        if (w == 0.f) continue;
        const float4 v = *reinterpret_cast<const float4*>(p.part_o + slot_row * p.D + d);
        a.x += w * v.x;
        a.y += w * v.y;
        a.z += w * v.z;
        a.w += w * v.w;
      }
      *reinterpret_cast<uint2*>(out + d) =
          make_uint2(pack_bf16x2(a.x * inv, a.y * inv), pack_bf16x2(a.z * inv, a.w * inv));
    }
    if (lane == 0 && p.lse) p.lse[row] = mx + lg2(L) * kLn2;
  }
}

}  // namespace pa
