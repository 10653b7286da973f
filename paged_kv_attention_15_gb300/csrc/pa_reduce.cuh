// Split-K combine kernels (included by the C-ABI unit only). Source: the
// MSLK pull request "[ROCm] Add FlyDSL paged-attention decode backend (dense
// + fp8) with benchmark" (Kernels: pa_decode_reduce, the split-K partial
// combine).
#pragma once

#include "pa_kernels.cuh"

namespace pa {

// ------------------------------------------------------------ row combine
// Pieces whose loads a warp keeps in flight at once. Four rather than
// eight keeps the kernels at most 64 registers (eight resident CTAs per SM):
// a row has two or three pieces at the benchmark workloads, and a launch of
// several thousand four-row CTAs then runs in one wave.
constexpr int kCombineGroup = 4;
// One warp combines the pieces k = 0..np-1 of one query row: M = max_k lse_k,
// w_k = exp(lse_k - M), out = sum_k w_k o_k / sum_k w_k, lse = M + ln sum_k w_k,
// in one online pass (running max, sums rescaled when it grows) that keeps
// the loads of KG pieces in flight. Pieces with lse = -inf weigh 0; a row
// whose pieces are all empty gets out = 0, lse = -inf; a piece whose lse is
// NaN (its work was cut short by a timed-out wait) makes the row NaN.
// o_row(k) points at piece k's D (<= 256; <= 128 unless WIDE) floats in
// global memory, read past L1 (other CTAs of the same grid may have written
// them); l_val(k) is its lse. Lane l owns columns 4l..4l+3 and, if WIDE,
// 128+4l..128+4l+3. Source: the
// MSLK pull request "[ROCm] Add FlyDSL paged-attention decode backend (dense
// + fp8) with benchmark" (Kernels: pa_decode_reduce, the split-K combine).
template <int KG, bool WIDE, typename ORow, typename LVal>
__device__ __forceinline__ void combine_row(int np, int D, ORow o_row, LVal l_val, __nv_bfloat16* out,
                                            float* lse_out, int lane, bool out_f16) {
  auto pack = [&](float lo, float hi) { return out_f16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi); };
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float LOG2E = 1.4426950408889634f;
  const int c0 = lane * 4, c1 = 128 + lane * 4;
  const bool h0 = c0 < D, h1 = WIDE && c1 < D;
  float m = NEG_INF, L = 0.f;
  bool poisoned = false;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  for (int k0 = 0; k0 < np; k0 += KG) {
    float lk[KG];
    float4 v0[KG], v1[KG];
#pragma unroll
    for (int j = 0; j < KG; ++j) {
      const bool in = k0 + j < np;
      lk[j] = in ? l_val(k0 + j) : NEG_INF;
      poisoned |= lk[j] != lk[j];
      const float* o = in ? o_row(k0 + j) : nullptr;
      v0[j] = in && h0 ? __ldcg(reinterpret_cast<const float4*>(o + c0)) : make_float4(0.f, 0.f, 0.f, 0.f);
      v1[j] = in && h1 ? __ldcg(reinterpret_cast<const float4*>(o + c1)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mc = m;
#pragma unroll
    for (int j = 0; j < KG; ++j) mc = fmaxf(mc, lk[j]);
    if (mc == NEG_INF) continue;
    const float so = m == NEG_INF ? 0.f : ex2((m - mc) * LOG2E);
    a0.x *= so; a0.y *= so; a0.z *= so; a0.w *= so;
    a1.x *= so; a1.y *= so; a1.z *= so; a1.w *= so;
    L *= so;
#pragma unroll
    for (int j = 0; j < KG; ++j) {
      if (lk[j] == NEG_INF) continue;
      const float w = ex2((lk[j] - mc) * LOG2E);
      a0.x += w * v0[j].x; a0.y += w * v0[j].y; a0.z += w * v0[j].z; a0.w += w * v0[j].w;
      a1.x += w * v1[j].x; a1.y += w * v1[j].y; a1.z += w * v1[j].z; a1.w += w * v1[j].w;
      L += w;
    }
    m = mc;
  }
  const float NaN = __int_as_float(0x7fffffff);
  const float inv = poisoned ? NaN : (L > 0.f ? 1.f / L : 0.f);
  if (h0)
    *reinterpret_cast<uint2*>(out + c0) =
        make_uint2(pack(a0.x * inv, a0.y * inv), pack(a0.z * inv, a0.w * inv));
  if (h1)
    *reinterpret_cast<uint2*>(out + c1) =
        make_uint2(pack(a1.x * inv, a1.y * inv), pack(a1.z * inv, a1.w * inv));
  if (lane == 0 && lse_out) *lse_out = poisoned ? NaN : (L > 0.f ? m + lg2(L) * kLn2 : NEG_INF);
}

// combine_row over a row of any D (a multiple of 4): 256 columns at a time
// (the weights are recomputed per chunk; they are the same every time).
template <int KG, typename ORow, typename LVal>
__device__ __forceinline__ void combine_row_any(int np, int D, ORow o_row, LVal l_val, __nv_bfloat16* out,
                                                float* lse_out, int lane, bool out_f16) {
  if (D <= 128) {
    combine_row<KG, false>(np, D, o_row, l_val, out, lse_out, lane, out_f16);
    return;
  }
  for (int c = 0; c < D; c += 256)
    combine_row<KG, true>(
        np, D - c < 256 ? D - c : 256, [&](int k) { return o_row(k) + c; }, l_val, out + c,
        c == 0 ? lse_out : nullptr, lane, out_f16);
}


// Explicit splits: grid covers B*T*Hq rows, 4 rows (warps) per CTA.
__global__ void __launch_bounds__(128, 8) pa_reduce_splits_kernel(const __grid_constant__ ReduceParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * 4 + warp;
  const size_t rows = (size_t)p.B * p.T * p.Hq;
  if (row >= rows) return;
  const size_t base = row * p.num_splits;
  wait_prerequisite_grids();  // the partials come from the split kernel
  const float* po = p.part_o + base * p.D;
  const float* pl = p.part_lse + base;
  const int D = p.D;
  combine_row_any<kCombineGroup>(
      p.num_splits, D, [&](int k) { return po + (size_t)k * D; }, [&](int k) { return __ldcg(pl + k); },
      p.out + row * D, p.lse ? p.lse + row : nullptr, lane, p.out_f16 != 0);
}

// Balanced launch: grid (units, ceil(M / 4)); warp w of CTA (u, y) combines
// row 4y + w of unit u = b * NHG + hg from the pieces that the split CTAs
// i0..i1 covering the unit wrote to slots u + i. Units wholly inside one
// CTA's share, and sequences with no keys, were written by the split kernel.
__global__ void __launch_bounds__(128, 8) pa_reduce_balanced_kernel(const __grid_constant__ ReduceParams p) {
  __shared__ long long s_sum[2][4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  const int b = u / p.NHG, hg = u % p.NHG;
  const int cap = p.max_blocks * p.P;
  int cb = __ldg(p.context_lens + b);  // (issued with the loop's loads: one round trip)
  long long before = 0, total = 0;
  for (int i = threadIdx.x; i < p.B; i += 128) {
    int c = __ldg(p.context_lens + i);
    c = c < 0 ? 0 : (c > cap ? cap : c);
    const long long nv = unit_vpages(c, p.P, p.tidar, p.item_w);
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
  cb = cb < 0 ? 0 : (cb > cap ? cap : cb);
  const long long nvb = unit_vpages(cb, p.P, p.tidar, p.item_w);
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
  combine_row_any<kCombineGroup>(
      i1 - i0 + 1, D, [&](int k) { return po + ((size_t)(u + i0 + k) * M + rho) * D; },
      [&](int k) {
        // A CTA whose share is empty wrote nothing; with at least as many
        // flattened pages as CTAs every share holds a page.
        const long long i = i0 + k;
        return (N >= G64 || (N * i / G64) < (N * (i + 1) / G64)) ? __ldcg(pl + (size_t)(u + i) * M + rho) : NEG_INF;
      },
      p.out + row * D, p.lse ? p.lse + row : nullptr, lane, p.out_f16 != 0);
}

}  // namespace pa
