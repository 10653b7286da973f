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
// Hkv rows of new tokens (contiguous in the source and in the cache slot)
// in 16-byte chunks; for fp8 a row's amax is a packed bf16 magnitude
// maximum and a shuffle reduction over the lanes holding the row,
// scale = amax / 448 and y = x / scale are correctly rounded float32
// quotients (two per instruction in the f32x2 arithmetic), and
// cvt.rn.satfinite makes the codes.
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

// Packed float32 pairs (the f32x2 arithmetic of sm_100 and later: two IEEE
// single-precision operations per instruction, subnormals kept).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2_rn(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2_rn(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fma2_rm(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// Per 16-bit half, the larger magnitude of two bf16 pairs (the sign bits of
// the result are the XOR of the inputs' and are cleared by the caller).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two correctly rounded quotients a / b at once, from r = RN(1/b) and
// nb = -b: Markstein's correction as in div_rn_by, with the remainder
// formed as a - q b (exact, as there) under rounding toward -inf, so that
// an exactly zero remainder is -0 and a = +0 / -0 still yield +0 / -0.
__device__ __forceinline__ uint64_t div2_rn_by(uint64_t a, uint64_t nb, uint64_t r) {
  const uint64_t q0 = mul2_rn(a, r);
  const uint64_t t = fma2_rm(q0, nb, a);
  return fma2_rn(t, r, q0);
}

// One wave of resident blocks; each warp step takes TPW consecutive tasks
// (kv, b, t). A task's Hkv rows are Hkv * D contiguous elements in k_new
// and in the cache slot. Lane pieces of E contiguous elements (E = 8, one
// 16-byte load, for bf16; E = 16 for fp8, so that the per-row work of the
// quantiser is shared by fewer lanes): piece c = 32 i + lane. A step keeps
// U = TPW R pieces per lane in flight before any store: R rounds of one task
// (TPW = 1), or, when a task has at most R rounds, all rounds of TPW tasks,
// whose payload loads all go out before the first slot lookup.
// Head h owns the L = D / E pieces [h L, (h + 1) L): for fp8 its amax is a
// shuffle reduction over those L lanes.
template <bool FP8, int D, int TPW, int R>
__global__ void __launch_bounds__(256) pa_kv_append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int E = FP8 ? 16 : 8;
  constexpr int V = E / 8;      // 16-byte loads per piece
  constexpr int L = D / E;
  constexpr int U = TPW * R;    // pieces in flight per lane
  const int lane = threadIdx.x & 31;
  const int pieces = p.Hkv * L;
  const int iters = (pieces + 31) / 32;  // rounds of a task (<= R when TPW > 1)
  const int cap = p.max_blocks * p.P;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int groups = (p.tasks + TPW - 1) / TPW;
  for (int grp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); grp < groups; grp += nwarps) {
    const uint4* src[TPW];
    int bb[TPW], tt[TPW], kvs[TPW];
#pragma unroll
    for (int s = 0; s < TPW; ++s) {
      const int task = min(grp * TPW + s, p.tasks - 1);  // (a task past the end is not loaded)
      const int kb = (int)div_by((uint32_t)task, p.mT, p.lT);
      tt[s] = task - kb * p.T;
      kvs[s] = (int)div_by((uint32_t)kb, p.mB, p.lB);
      bb[s] = kb - kvs[s] * p.B;
      src[s] = reinterpret_cast<const uint4*>((kvs[s] ? p.v_new : p.k_new) +
                                              ((size_t)bb[s] * p.T + tt[s]) * p.Hkv * D);
    }
    bool ok[TPW];
    size_t row0[TPW];  // cache row of head 0
    for (int i0 = 0; i0 < iters; i0 += U) {  // (one pass when TPW > 1)
      // The payload loads go out first; the slot lookups overlap them.
      uint4 x[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int s = u / R;
        const int rd = TPW > 1 ? u % R : i0 + u;
        const int pc = rd * 32 + lane;
        const bool live = rd < iters && pc < pieces && grp * TPW + s < p.tasks;
#pragma unroll
        for (int v = 0; v < V; ++v) x[u][v] = live ? __ldcs(src[s] + pc * V + v) : make_uint4(0, 0, 0, 0);
      }
      if (i0 == 0) {
#pragma unroll
        for (int s = 0; s < TPW; ++s) {
          int c = __ldg(p.context_lens + bb[s]);
          c = c < 0 ? 0 : (c > cap ? cap : c);
          const int j = c + tt[s];
          int page = -1, slot = 0;
          if (j < cap) {
            const int pi = p.lgP >= 0 ? j >> p.lgP : j / p.P;
            slot = p.lgP >= 0 ? j & (p.P - 1) : j - pi * p.P;
            page = __ldg(p.block_tables + (size_t)bb[s] * p.max_blocks + pi);
          }
          ok[s] = page >= 0 && page < p.num_pages && grp * TPW + s < p.tasks;  // warp-uniform
          row0[s] = ((size_t)page * p.P + slot) * p.Hkv;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int s = u / R;
        const int rd = TPW > 1 ? u % R : i0 + u;
        if (rd >= iters) continue;  // warp-uniform
        const int pc = rd * 32 + lane;
        const bool mine = ok[s] && pc < pieces;
        if constexpr (!FP8) {
          if (mine)
            reinterpret_cast<uint4*>(static_cast<uint16_t*>(kvs[s] ? p.v_cache : p.k_cache) + row0[s] * D)[pc] =
                x[u][0];
        } else {
          uint32_t w[8];
#pragma unroll
          for (int v = 0; v < V; ++v) {
            w[4 * v] = x[u][v].x;
            w[4 * v + 1] = x[u][v].y;
            w[4 * v + 2] = x[u][v].z;
            w[4 * v + 3] = x[u][v].w;
          }
          // Element 2e is the low half of w[e], element 2e + 1 the high half.
          uint32_t m2 = absmax_bf16x2(w[0], w[1]);
#pragma unroll
          for (int e = 2; e < 8; ++e) m2 = absmax_bf16x2(m2, w[e]);
          m2 &= 0x7FFF7FFFu;
          float amax = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
#pragma unroll
          for (int o = L / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          // scale = RN(amax / 448); y = RN(x / scale), both correctly rounded.
          // Rows with amax < 2^-60 take IEEE divisions: there the remainders
          // of the FMA path could fall below the normal range (any y whose
          // code is not zero keeps every intermediate normal above it).
          const bool tiny = amax < 0x1p-60f;
          const float scale = amax > 0.f ? (tiny ? __fdiv_rn(amax, 448.f) : div_rn_by(amax, 448.f, kRcp448)) : 1.f;
          float y[E];
          if (!tiny) {
            const float rcp = __frcp_rn(scale);
            const uint64_t r2 = pack2(rcp, rcp), nb2 = pack2(-scale, -scale);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint64_t a = pack2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
              unpack2(div2_rn_by(a, nb2, r2), y[2 * e], y[2 * e + 1]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              y[2 * e] = __fdiv_rn(__uint_as_float(w[e] << 16), scale);
              y[2 * e + 1] = __fdiv_rn(__uint_as_float(w[e] & 0xFFFF0000u), scale);
            }
          }
          uint32_t q[E / 4];
#pragma unroll
          for (int e = 0; e < E / 4; ++e) {
            const uint32_t lo = f32x2_to_e4m3x2(y[4 * e], y[4 * e + 1]);
            const uint32_t hi = f32x2_to_e4m3x2(y[4 * e + 2], y[4 * e + 3]);
            q[e] = lo | (hi << 16);
          }
          if (mine) {
            uint8_t* cache = static_cast<uint8_t*>(kvs[s] ? p.v_cache : p.k_cache);
            reinterpret_cast<uint4*>(cache + row0[s] * D)[pc] = make_uint4(q[0], q[1], q[2], q[3]);
            if (pc % L == 0) (kvs[s] ? p.v_scale : p.k_scale)[row0[s] + pc / L] = scale;
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
template <bool FP8, int D, int TPW, int R>
int blocks_per_sm() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pa_kv_append_kernel<FP8, D, TPW, R>, 256, 0) != cudaSuccess ||
      n < 1)
    n = 1;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <bool FP8, int D, int TPW, int R>
cudaError_t launch_t(const AppendParams& p, cudaStream_t stream) {
  // One wave of resident blocks (fewer when there are fewer task groups).
  const long long resident = (long long)(sm_count() > 0 ? sm_count() : 1) * blocks_per_sm<FP8, D, TPW, R>();
  long long blocks = ((long long)(p.tasks + TPW - 1) / TPW + 7) / 8;
  if (blocks > resident) blocks = resident;
  pa_kv_append_kernel<FP8, D, TPW, R><<<dim3((unsigned)blocks), dim3(256), 0, stream>>>(p);
  return cudaGetLastError();
}

// Tasks per warp step and slots per task. When the call has at least as
// many tasks as a wave of resident warps: 16-bit rows take all rounds of
// four tasks (one round each), of two (two rounds each), else four rounds
// of one task at a time; fp8 rows (whose quantiser holds more registers per
// piece) two one-round tasks, else two rounds of one task (more tasks per
// step measured slower: the registers cut the resident warps). Calls with
// fewer tasks (a decode step's append) keep one task per warp step, so that
// every task has a warp of its own.
template <bool FP8, int D>
cudaError_t launch_d(const AppendParams& p, cudaStream_t stream) {
  constexpr int E = FP8 ? 16 : 8;
  const long long rounds = ((long long)p.Hkv * (D / E) + 31) / 32;
  const long long wave =
      (long long)(sm_count() > 0 ? sm_count() : 1) * blocks_per_sm<FP8, D, 1, FP8 ? 2 : 4>() * 8;
  const bool few = p.tasks < wave;
  if constexpr (FP8) {
    if (rounds == 1) return few ? launch_t<FP8, D, 1, 1>(p, stream) : launch_t<FP8, D, 2, 1>(p, stream);
    return launch_t<FP8, D, 1, 2>(p, stream);
  } else {
    if (rounds == 1) return few ? launch_t<FP8, D, 1, 1>(p, stream) : launch_t<FP8, D, 4, 1>(p, stream);
    if (rounds == 2) return few ? launch_t<FP8, D, 1, 2>(p, stream) : launch_t<FP8, D, 2, 2>(p, stream);
    return launch_t<FP8, D, 1, 4>(p, stream);
  }
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
