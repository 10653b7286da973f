// KV-cache append: the step before a decode writes each sequence's new K/V
// rows into their page slots, and for an fp8 cache quantises each row
// (token, kv head) with its own scale.
//
// The paged cache with per-sequence block tables is the problem of the ROCm
// blog page "Implementing a High-Performance Custom Diffusion Attention
// Kernel with FlyDSL" (introduction item 1); the fp8 format (OCP e4m3fn,
// symmetric per-token scale) is the MSLK pull request "[ROCm] Add FlyDSL
// paged-attention decode backend (dense + fp8) with benchmark" (Kernels;
// Other changes), whose review asks for scales computed when the cache is
// written.
//
// A plain streaming copy: HBM-bound, no tensor-core work. A warp moves the
// Hkv rows of one new token (contiguous in the source and in the cache slot)
// in 16-byte chunks; for fp8 a row's amax is a shuffle reduction over the
// D/8 lanes holding it, scale = amax / 448 and y = x / scale are correctly
// rounded float32 quotients, and cvt.rn.satfinite makes the codes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "pa_decode.h"
#include "pa_ptx.cuh"

namespace pa {

struct AppendParams {
  const uint16_t* k_new;  // bf16 bits [B, T, Hkv, D]
  const uint16_t* v_new;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* k_cache;  // [num_pages, P, Hkv, D] bf16 or e4m3fn
  void* v_cache;
  float* k_scale;  // fp8: [num_pages, P, Hkv]
  float* v_scale;
  int B, T, Hkv, P, max_blocks, num_pages;
  int lgP;     // log2(P) when P is a power of two, else -1
  int tasks;   // 2 * B * T: task = (kv * B + b) * T + t, the Hkv rows of one token of K or V
  uint32_t mT, mB;  // n / T and n / B as (umulhi(n, m) + n) >> l (round-up reciprocal)
  int lT, lB;
};

// n / d for 0 <= n < 2^31 from the precomputed m = floor(2^32 (2^l - d) / d) + 1,
// l = ceil(log2 d) (T. Granlund, P. Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994).
__device__ __forceinline__ uint32_t div_by(uint32_t n, uint32_t m, int l) {
  return (uint32_t)(((uint64_t)__umulhi(n, m) + n) >> l);
}

// RN(1/448) in float32 (the correctly rounded reciprocal of 448).
constexpr float kRcp448 = 0x1.24924ap-9f;

// Correctly rounded a / b from r = RN(1/b) by Markstein's theorem
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with q = RN(a r)
// the remainder a - q b is exact in one FMA, and RN(q + (a - q b) r) =
// RN(a / b) while no intermediate overflows or underflows. The remainder is
// formed as -(q b - a) so that a = -0 yields -0 (as IEEE division does).
__device__ __forceinline__ float div_rn_by(float a, float b, float r) {
  const float q0 = __fmul_rn(a, r);
  const float t = __fmaf_rn(q0, b, -a);
  return __fmaf_rn(-t, r, q0);
}

// One wave of resident blocks; warps take tasks (kv, b, t) in turn. A
// task's Hkv rows are Hkv * D contiguous elements in k_new and in the cache
// slot. Lane pieces of E contiguous elements (E = 8, one 16-byte load, for
// bf16; E = 16 for fp8, so that the per-row work of the quantiser is shared
// by fewer lanes): piece c = 32 i + lane, several pieces of a lane in flight
// before any store. Head h owns the L = D / E pieces [h L, (h + 1) L): for
// fp8 its amax is a shuffle reduction over those L lanes.
template <bool FP8, int D>
__global__ void __launch_bounds__(256) pa_kv_append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int E = FP8 ? 16 : 8;
  constexpr int V = E / 8;      // 16-byte loads per piece
  constexpr int L = D / E;
  constexpr int U = FP8 ? 2 : 4;  // pieces in flight per lane
  const int lane = threadIdx.x & 31;
  const int pieces = p.Hkv * L;
  const int iters = (pieces + 31) / 32;
  const int cap = p.max_blocks * p.P;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int task = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < p.tasks; task += nwarps) {
    const int kb = (int)div_by((uint32_t)task, p.mT, p.lT);
    const int t = task - kb * p.T;
    const int kv = (int)div_by((uint32_t)kb, p.mB, p.lB);
    const int b = kb - kv * p.B;
    const uint4* src = reinterpret_cast<const uint4*>((kv ? p.v_new : p.k_new) + ((size_t)b * p.T + t) * p.Hkv * D);
    const int32_t* bt = p.block_tables + (size_t)b * p.max_blocks;
    int c = __ldg(p.context_lens + b);
    c = c < 0 ? 0 : (c > cap ? cap : c);
    const int j = c + t;
    bool ok = false;
    size_t row0 = 0;  // cache row of head 0
    for (int i0 = 0; i0 < iters; i0 += U) {
      // The payload loads go out first; the slot lookup overlaps them.
      uint4 x[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int pc = (i0 + u) * 32 + lane;
#pragma unroll
        for (int v = 0; v < V; ++v) {
          x[u][v] = make_uint4(0, 0, 0, 0);
          if (i0 + u < iters && pc < pieces) x[u][v] = __ldcs(src + pc * V + v);
        }
      }
      if (i0 == 0) {
        int page = -1, slot = 0;
        if (j < cap) {
          const int pi = p.lgP >= 0 ? j >> p.lgP : j / p.P;
          slot = p.lgP >= 0 ? j & (p.P - 1) : j - pi * p.P;
          page = __ldg(bt + pi);
        }
        ok = page >= 0 && page < p.num_pages;  // warp-uniform
        row0 = ((size_t)page * p.P + slot) * p.Hkv;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (i0 + u >= iters) break;  // warp-uniform
        const int pc = (i0 + u) * 32 + lane;
        const bool mine = ok && pc < pieces;
        if constexpr (!FP8) {
          if (mine) reinterpret_cast<uint4*>(static_cast<uint16_t*>(kv ? p.v_cache : p.k_cache) + row0 * D)[pc] = x[u][0];
        } else {
        float f[E];
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const uint32_t w[4] = {x[u][v].x, x[u][v].y, x[u][v].z, x[u][v].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            f[8 * v + 2 * e] = __uint_as_float(w[e] << 16);
            f[8 * v + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
          }
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
        for (int o = L / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        // scale = RN(amax / 448); y = RN(x / scale), both correctly rounded.
        // Rows with amax < 2^-60 take IEEE divisions: there the remainders
        // of the FMA path could fall below the normal range (any y whose
        // code is not zero keeps every intermediate normal above it).
        const bool tiny = amax < 0x1p-60f;
        const float scale = amax > 0.f ? (tiny ? __fdiv_rn(amax, 448.f) : div_rn_by(amax, 448.f, kRcp448)) : 1.f;
        const float rcp = __frcp_rn(scale);
        float y[E];
        if (!tiny) {
#pragma unroll
          for (int e = 0; e < E; ++e) y[e] = div_rn_by(f[e], scale, rcp);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) y[e] = __fdiv_rn(f[e], scale);
        }
        uint32_t q[E / 4];
#pragma unroll
        for (int e = 0; e < E / 4; ++e) {
          const uint32_t lo = f32x2_to_e4m3x2(y[4 * e], y[4 * e + 1]);
          const uint32_t hi = f32x2_to_e4m3x2(y[4 * e + 2], y[4 * e + 3]);
          q[e] = lo | (hi << 16);
        }
        if (mine) {
          uint8_t* cache = static_cast<uint8_t*>(kv ? p.v_cache : p.k_cache);
          reinterpret_cast<uint4*>(cache + row0 * D)[pc] = make_uint4(q[0], q[1], q[2], q[3]);
          if (pc % L == 0) (kv ? p.v_scale : p.k_scale)[row0 + pc / L] = scale;
        }
        }
      }
    }
  }
}

namespace {

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

// Multiplier and shift of div_by for a divisor d >= 1.
void magic(uint32_t d, uint32_t* m, int* l) {
  int s = 0;
  while ((1ull << s) < d) ++s;
  *l = s;
  *m = (uint32_t)(((1ull << 32) * ((1ull << s) - d)) / d + 1);
}

// Per-device values cached by any thread (idempotent: a race only repeats
// the query).
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Resident blocks per SM of an instance, asked of the runtime once per device.
template <bool FP8, int D>
int blocks_per_sm() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pa_kv_append_kernel<FP8, D>, 256, 0) != cudaSuccess || n < 1)
    n = 1;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <bool FP8, int D>
cudaError_t launch_d(const AppendParams& p, cudaStream_t stream) {
  // One wave of resident blocks (fewer when there are fewer tasks).
  const long long resident = (long long)(sm_count() > 0 ? sm_count() : 1) * blocks_per_sm<FP8, D>();
  long long blocks = (p.tasks + 7) / 8;
  if (blocks > resident) blocks = resident;
  pa_kv_append_kernel<FP8, D><<<dim3((unsigned)blocks), dim3(256), 0, stream>>>(p);
  return cudaGetLastError();
}

template <bool FP8>
cudaError_t launch(int D, const AppendParams& p, cudaStream_t stream) {
  if (D == 64) return launch_d<FP8, 64>(p, stream);
  if (D == 128) return launch_d<FP8, 128>(p, stream);
  return launch_d<FP8, 256>(p, stream);
}

pa_status run_append(bool fp8, const void* k_new, const void* v_new, const int32_t* block_tables,
                     const int32_t* context_lens, const pa_shape* s, void* k_cache, void* v_cache, float* k_scale,
                     float* v_scale, pa_stream_t stream) {
  if (!s) return PA_ERR_INVALID_ARG;
  if (s->batch < 0 || s->q_tokens < 1 || s->num_kv_heads < 1 || s->page_size < 1 || s->num_pages < 1 ||
      s->max_blocks_per_seq < 1)
    return PA_ERR_INVALID_ARG;
  if ((int64_t)s->max_blocks_per_seq * s->page_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  const int D = s->head_dim;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !block_tables || !context_lens || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale))) return PA_ERR_INVALID_ARG;
  if (s->batch == 0) return PA_OK;
  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.B = s->batch;
  p.T = s->q_tokens;
  p.Hkv = s->num_kv_heads;
  p.P = s->page_size;
  p.max_blocks = s->max_blocks_per_seq;
  p.num_pages = s->num_pages;
  if (2LL * s->batch * s->q_tokens > INT32_MAX || (long long)s->q_tokens * s->num_kv_heads * D > INT32_MAX)
    return PA_ERR_INVALID_ARG;
  p.tasks = 2 * s->batch * s->q_tokens;
  magic(s->q_tokens, &p.mT, &p.lT);
  magic(s->batch, &p.mB, &p.lB);
  p.lgP = (s->page_size & (s->page_size - 1)) == 0 ? __builtin_ctz((unsigned)s->page_size) : -1;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t err = fp8 ? launch<true>(D, p, st) : launch<false>(D, p, st);
  return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

extern "C" {

pa_status pa_kv_append(const void* k_new, const void* v_new, const int32_t* block_tables,
                       const int32_t* context_lens, const pa_shape* shape, void* k_cache, void* v_cache,
                       pa_stream_t stream) {
  return pa::run_append(false, k_new, v_new, block_tables, context_lens, shape, k_cache, v_cache, nullptr, nullptr,
                        stream);
}

pa_status pa_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* block_tables,
                           const int32_t* context_lens, const pa_shape* shape, uint8_t* k_cache, uint8_t* v_cache,
                           float* k_scale, float* v_scale, pa_stream_t stream) {
  return pa::run_append(true, k_new, v_new, block_tables, context_lens, shape, k_cache, v_cache, k_scale, v_scale,
                        stream);
}

}  // extern "C"
