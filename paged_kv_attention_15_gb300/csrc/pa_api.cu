// C ABI of the paged-KV decode engine: argument checks, work scheduling,
// TMA descriptor encoding and kernel launches. See include/pa_decode.h.
#include "pa_decode.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pa_launch.h"
#include "pa_reduce.cuh"

namespace {

using pa::ReduceParams;
using pa::SplitKernel;
using pa::SplitParams;

// Error flags written by the kernels (one word per device: each device has
// its own copy of a module-scope __device__ variable).
__device__ int g_pa_err_flags;

constexpr int kMaxDevices = 64;
constexpr int kKernelSlots = 16;

// Per-device values looked up once; `ready` publishes them (release) to
// threads that read it (acquire) without taking the lock.
struct DeviceState {
  std::atomic<bool> ready;
  int sms;
  int smem_optin;
  int* err_flags;
  std::atomic<const void*> smem_set[kKernelSlots];  // kernels prepared for launch (setup_kernel)
};

DeviceState g_dev[kMaxDevices];  // zero-initialised (static storage)
std::mutex g_mu;

// One-shot events armed by pa_decode_profile_events for this thread's next call.
thread_local cudaEvent_t t_ev_start = nullptr;
thread_local cudaEvent_t t_ev_split = nullptr;

enum class Kind { kBf16, kFp8, kTidar, kF16 };

pa_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  DeviceState& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PA_ERR_CUDA;
      if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return PA_ERR_CUDA;
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_pa_err_flags) != cudaSuccess) return PA_ERR_CUDA;
      d.err_flags = static_cast<int*>(ptr);
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return PA_OK;
}

// Prepares a kernel for launch, once per device: raises its dynamic
// shared-memory limit and, for a kernel that moves registers between its
// warpgroups, checks that it was built with the launch registers its split
// draws on (with fewer, a setmaxnreg.inc would wait for registers that never
// come; the call is refused instead).
pa_status setup_kernel(DeviceState* d, const SplitKernel& k) {
  if (k.launch_regs > 0) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, k.fn) != cudaSuccess) return PA_ERR_CUDA;
    if (a.numRegs < k.launch_regs) return PA_ERR_UNSUPPORTED;
  }
  return cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, d->smem_optin) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status ensure_kernel_ready(DeviceState* d, const SplitKernel& k) {
  for (int i = 0; i < kKernelSlots; ++i)
    if (d->smem_set[i].load(std::memory_order_acquire) == k.fn) return PA_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < kKernelSlots; ++i) {
    const void* cur = d->smem_set[i].load(std::memory_order_relaxed);
    if (cur == k.fn) return PA_OK;
    if (cur == nullptr) {
      const pa_status st = setup_kernel(d, k);
      if (st == PA_OK) d->smem_set[i].store(k.fn, std::memory_order_release);
      return st;
    }
  }
  return setup_kernel(d, k);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Rank-R map (R = 4 or 5), dims innermost first, strides in bytes for dims
// 1..R-1, 128-byte swizzle.
template <int R>
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[R],
              const uint64_t (&strides)[R - 1], const uint32_t (&box)[R]) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[R], gs[R - 1];
  cuuint32_t bx[R], es[R];
  for (int i = 0; i < R; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i < R - 1) gs[i] = strides[i];
  }
  return fn(m, dt, R, const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Shape checks shared by every entry point.
pa_status check_shape(const pa_shape* s, Kind kind) {
  if (!s) return PA_ERR_INVALID_ARG;
  if (s->batch < 0 || s->q_tokens < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 || s->head_dim < 1 ||
      s->page_size < 1 || s->num_pages < 1 || s->max_blocks_per_seq < 1)
    return PA_ERR_INVALID_ARG;
  if (s->num_q_heads % s->num_kv_heads) return PA_ERR_INVALID_ARG;
  if ((int64_t)s->max_blocks_per_seq * s->page_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  const int D = s->head_dim;
  if (kind == Kind::kFp8) {
    if (D != 128 && D != 256) return PA_ERR_UNSUPPORTED;
  } else if (D != 64 && D != 128 && D != 256) {
    return PA_ERR_UNSUPPORTED;
  }
  if (!pow2_in(s->page_size, 16, 256)) return PA_ERR_UNSUPPORTED;
  const int64_t M = (int64_t)(s->num_q_heads / s->num_kv_heads) * s->q_tokens;
  if (M > 64) return PA_ERR_UNSUPPORTED;
  if (M > 32 && (kind == Kind::kFp8 || D == 256)) return PA_ERR_UNSUPPORTED;  // four row tiles: D <= 128, bf16
  return PA_OK;
}

SplitKernel pick_kernel(Kind kind, int D, int MT, int TSL, int CW) {
  if (kind == Kind::kFp8) return pa::split_kernel_fp8(D, MT, TSL, CW);
  if (kind == Kind::kF16) return pa::split_kernel_f16(D, MT, TSL, CW);
  return pa::split_kernel_bf16(D, MT, TSL, CW);
}

// Work-unit geometry: H2 kv heads per CTA unit, their M = H2 * G * T query
// rows in MT m16 tiles, TS = 64 / H2 tokens per stage, TSL tokens per warp.
// Token-major tcgen05 kernel: M = N rows, TS = 128 / H2 tokens per stage.
// Query-row-major tcgen05 kernel: M = 64 rows, TS = 64 / H2.
struct Geom {
  int GT, H2, NHG, M, MT, TS, TSL, BR, lbr, TP, ilv;
  int path;          // kernel: kPathWarp, kPathUmma, kPathQrow or kPathPair
  int chunk_boxes;   // 1: one copy per page and 128-byte column chunk (query-row kernel)
  SplitKernel k;
};

// Decode kernels (pa_decode_set_kernel_path / pa_decode_kernel_for).
constexpr int kPathAuto = 0, kPathWarp = 1, kPathUmma = 2, kPathQrow = 3, kPathPair = 4;
constexpr int kPairItemPages = 8, kItemPages = 4;  // Plan::item_w of the paired-role kernel, of the others

// Which decode kernel a call may use: automatic, the warp-level MMA kernel
// only, or one of the tcgen05 kernels wherever it has an instance.
std::atomic<int> g_kernel_path{kPathAuto};

// How the balanced schedule's pieces are combined: a separate reduce kernel
// (0), or fused into the warp-level split kernel (1: its last CTA to finish a
// unit's piece combines the unit).
std::atomic<int> g_combine_mode{0};

int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// pair: the split kernel with paired consumer roles (four pairs, each an S
// warp and a PV warp), laid out like four consumer warps.
bool geom_for(const pa_shape* s, Kind kind, int H2, Geom* g, bool pair = false) {
  const int G = s->num_q_heads / s->num_kv_heads, T = s->q_tokens, P = s->page_size, D = s->head_dim;
  const int GT = G * T, M = H2 * GT;
  if (M > 64 || s->num_kv_heads % H2) return false;
  // With several heads per unit, a head's rows must fill whole m16 tiles or
  // share one evenly.
  if (H2 > 1 && (GT < 16 ? 16 % GT : GT % 16)) return false;
  const int MT = M <= 16 ? 1 : (M <= 32 ? 2 : 4);  // rows past M are masked
  // Eight consumer warps (two per row tile, splitting its tokens) where
  // such an instance is built, else four.
  const bool fp8 = kind == Kind::kFp8;
  const int cap_rows = pa::stage_rows(D * (fp8 ? 1 : 2), fp8);
  // The draft block's scratch stage lands TP rows of each of the unit's
  // heads in one stage tile.
  if (kind == Kind::kTidar && (T + 7) / 8 * 8 * H2 > cap_rows) return false;
  const int HT = GT >= 16 ? 1 : (16 / GT < H2 ? 16 / GT : H2);  // heads in a row tile
  SplitKernel k{nullptr, 0, 0, 0};
  int TS = 0, TSL = 0, ilv = 1;
  for (int CW = pair ? pa::kConsumerWarps : 8; CW >= pa::kConsumerWarps && !k.fn; CW /= 2) {
    const int NGW = CW / MT;
    if (NGW < 1 || NGW % HT) continue;
    const int NSL = NGW / HT;
    // Stage rows: the instance's capacity when a warp's token slice allows
    // it, else 64.
    for (int rows = cap_rows; rows >= (cap_rows < 64 ? cap_rows : 64) && !k.fn; rows /= 2) {
      TS = rows / H2;
      if (TS % NSL) continue;
      const int base = TS / NSL;  // tokens per warp if every slice group took every stage
      // Slice groups take 32 (else `base`) tokens of every ilv-th stage
      // where such an instance is built (more independent MMA chains per
      // warp, fewer softmax reductions per token); NSL / ilv slices per stage.
      for (TSL = base < 32 ? 32 : base; TSL >= base; TSL /= 2) {
        ilv = TSL / base;
        if (TSL != 16 && TSL != 32 && TSL != 64) continue;
        if (ilv > NSL || NSL % ilv) continue;
        k = pair ? (kind == Kind::kFp8 ? pa::pair_kernel_fp8(D, MT, TSL)
                                       : pa::pair_kernel_16(D, kind == Kind::kF16, MT, TSL))
                 : pick_kernel(kind, D, MT, TSL, CW);
        if (k.fn) break;
      }
    }
  }
  if (!k.fn) return false;
  g->ilv = ilv;
  g->GT = GT;
  g->H2 = H2;
  g->NHG = s->num_kv_heads / H2;
  g->M = M;
  g->path = pair ? kPathPair : kPathWarp;
  g->chunk_boxes = 0;
  g->MT = MT;
  g->TS = TS;
  g->TSL = TSL;
  g->BR = P < TS ? P : TS;
  g->lbr = ilog2(g->BR);
  g->TP = (T + 7) / 8 * 8;
  g->k = k;
  return true;
}

// tcgen05 kernel geometry: G * T query rows per kv head (16 or 32), the
// most kv heads per unit (up to 4) whose N = H2 * G * T rows have an
// instance; a stage holds TS = 128 / H2 tokens of each head.
bool geom_umma(const pa_shape* s, Kind kind, Geom* g) {
  const int G = s->num_q_heads / s->num_kv_heads, T = s->q_tokens, P = s->page_size, D = s->head_dim;
  const int GT = G * T;
  if (GT != 16 && GT != 32) return false;
  for (int H2 = 4; H2 >= 1; H2 /= 2) {
    const int N = H2 * GT;
    if (s->num_kv_heads % H2 || N > 64) continue;
    const int TS = 128 / H2, TP = (T + 7) / 8 * 8;
    if (kind == Kind::kTidar && TP > TS) continue;
    const SplitKernel k = kind == Kind::kFp8 ? pa::umma_kernel_fp8(D, GT, N)
                                             : pa::umma_kernel_16(D, kind == Kind::kF16, GT, N);
    if (!k.fn) continue;
    g->GT = GT;
    g->H2 = H2;
    g->NHG = s->num_kv_heads / H2;
    g->M = N;
    g->MT = 0;
    g->TS = TS;
    g->TSL = 0;
    g->BR = P < TS ? P : TS;
    g->lbr = ilog2(g->BR);
    g->TP = TP;
    g->ilv = 1;
    g->path = kPathUmma;
    g->chunk_boxes = 0;
    g->k = k;
    return true;
  }
  return false;
}

// Query-row-major tcgen05 kernel geometry: 16-bit caches, D = 128; units of
// 128 query rows (four kv heads of G * T = 32 rows: one 16-token page box
// of the four heads per 64-key-row stage) where the kv heads group by four,
// else of 64 rows (two kv heads of 32 rows, or one of 64; stages of 64 key
// rows copied per page and 128-byte chunk, page boxes of at least 16 rows);
// the draft scratch in one box whose key rows fill whole 16-row MMA steps.
bool geom_qrow(const pa_shape* s, Kind kind, Geom* g) {
  if (kind == Kind::kFp8) return false;
  const int G = s->num_q_heads / s->num_kv_heads, T = s->q_tokens, P = s->page_size, D = s->head_dim;
  const int GT = G * T;
  int H2 = GT == 32 ? 2 : (GT == 64 ? 1 : 0);
  int M = 64;
  if (GT == 32 && s->num_kv_heads % 4 == 0 && pa::qrow_kernel_16(D, kind == Kind::kF16, 4, 128).fn) {
    H2 = 4;
    M = 128;
  }
  if (H2 == 0 || s->num_kv_heads % H2) return false;
  const int TS = 64 / H2, BR = P < TS ? P : TS;
  if (BR < 16) return false;
  int TP = (T + 15) / 16 * 16;
  if (H2 >= 2 && T <= 8) TP = 8;
  if (kind == Kind::kTidar && TP * H2 > 64) return false;
  const SplitKernel k = pa::qrow_kernel_16(D, kind == Kind::kF16, H2, M);
  if (!k.fn) return false;
  g->GT = GT;
  g->H2 = H2;
  g->NHG = s->num_kv_heads / H2;
  g->M = M;
  g->MT = 0;
  g->TS = TS;
  g->TSL = 0;
  g->BR = BR;
  g->lbr = ilog2(BR);
  g->TP = TP;
  g->ilv = 1;
  g->path = kPathQrow;
  g->chunk_boxes = M == 64 ? 1 : 0;
  g->k = k;
  return true;
}

// Automatic choice: for fp8 caches the paired-role warp-level kernel
// (measured faster on the fp8 workload), else the single-role one; a tcgen05
// kernel on request.
int wanted_path() { return g_kernel_path.load(std::memory_order_relaxed); }

// One kv head per unit, or more while a page's box stays under 16 KB: a
// 16-row page of one head is a 4 KB copy, too small to keep enough bytes in
// flight per SM.
pa_status pick_geometry(const pa_shape* s, Kind kind, Geom* out, int path = -1) {
  const int want = path >= 0 ? path : wanted_path();
  if (want == kPathUmma && geom_umma(s, kind, out)) return PA_OK;
  if (want == kPathQrow && geom_qrow(s, kind, out)) return PA_OK;
  // The paired-role kernel where it has an instance for the shape, else the
  // single-role warp-level kernel.
  // From the smallest unit with an instance (one kv head for the
  // single-role kernel; the paired kernel's 16-bit instances start at 64
  // query rows), grow it while its page box stays under 16 KB.
  const int e = kind == Kind::kFp8 ? 1 : 2;
  auto search = [&](bool pair, Geom* best) {
    bool have = false;
    for (int cand = 1; cand <= 8; cand *= 2) {
      if (have && (long)best->BR * best->H2 * s->head_dim * e >= 16384) break;
      Geom g;
      if (!geom_for(s, kind, cand, &g, pair)) {
        if (have) break;
        continue;
      }
      *best = g;
      have = true;
    }
    return have;
  };
  const bool pair = want == kPathPair || (want == kPathAuto && kind == Kind::kFp8);
  if (pair && search(true, out)) return PA_OK;
  return search(false, out) ? PA_OK : PA_ERR_UNSUPPORTED;
}

// The launch plan of a call: mode, grid and workspace.
struct Plan {
  Geom geo;
  bool balanced = false;  // equal shares of the flattened pages, one CTA per SM
  int splits = 1;         // explicit mode
  int grid = 0;           // balanced mode CTAs
  size_t smem = 0;
  size_t ws_bytes = 0;
  size_t part_lse_off = 0;
  size_t count_off = 0;   // balanced mode: per-unit arrival counters of the fused combine
  int item_w = 0;         // balanced mode: virtual pages charged per work item (SplitParams::item_w)
};

// path: the kernel selection to plan for (-1: the current setting).
pa_status make_plan(const pa_shape* s, Kind kind, int num_splits, DeviceState* d, Plan* plan, int path = -1) {
  Geom geo;
  pa_status st = pick_geometry(s, kind, &geo, path);
  if (st != PA_OK) return st;
  const SplitKernel k = geo.k;
  const int B = s->batch, T = s->q_tokens, Hq = s->num_q_heads, D = s->head_dim;
  const int M = geo.M, units = B * geo.NHG;
  Plan p;
  p.geo = geo;
  // The fixed cost of a work item (Q load and conversion, merge, partial
  // write) in pages of the balanced schedule: on the paired-role kernel's fp8
  // workload a CTA's extra item cost about 3.3 us, some seven pages' worth
  // (8: split kernel 121.5 -> 118.8 us); 4 for the other kernels (gqa_d64
  // 63.5 -> 61.5 us, the other workloads unchanged).
  p.item_w = geo.path == kPathPair ? kPairItemPages : kItemPages;
  // A call too small to give every SM several pages gains nothing from the
  // weights, only more CTAs with empty shares.
  if ((long long)units * s->max_blocks_per_seq < 4LL * d->sms) p.item_w = 0;
  if (num_splits == 0) {
    const size_t smem = (size_t)k.smem_fixed + (size_t)(2 * B + 1) * 4;
    if (smem <= (size_t)d->smem_optin) {
      p.balanced = true;
      // One CTA per SM, but no more CTAs than the flattened pages can fill
      // (more would only add empty shares for the reduce to skip).
      const long long most =
          (long long)units * (s->max_blocks_per_seq + (kind == Kind::kTidar ? 1 : 0) + p.item_w);
      p.grid = most < d->sms ? (int)(most < 1 ? 1 : most) : d->sms;
      p.smem = smem;
      const size_t slots = (size_t)units + p.grid;
      p.part_lse_off = align256(slots * M * D * sizeof(float));
      p.count_off = p.part_lse_off + align256(slots * M * sizeof(float));
      p.ws_bytes = p.count_off + align256((size_t)units * sizeof(unsigned));
      *plan = p;
      return PA_OK;
    }
    // Too many sequences for the on-chip table: explicit splits that give
    // every SM about two CTAs.
    int S = (2 * d->sms + units - 1) / units;
    S = S < 1 ? 1 : (S > s->max_blocks_per_seq ? s->max_blocks_per_seq : S);
    num_splits = S;
  }
  if (num_splits > 65535) return PA_ERR_UNSUPPORTED;
  p.splits = num_splits;
  p.smem = (size_t)k.smem_fixed;
  if (p.smem > (size_t)d->smem_optin) return PA_ERR_UNSUPPORTED;
  if (num_splits > 1) {
    const size_t rows = (size_t)B * T * Hq * num_splits;
    p.part_lse_off = align256(rows * D * sizeof(float));
    p.ws_bytes = p.part_lse_off + align256(rows * sizeof(float));
  }
  *plan = p;
  return PA_OK;
}

struct CallArgs {
  Kind kind;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;
  const float* v_scale;
  const void* k_scratch;
  const void* v_scratch;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const pa_shape* shape;
  float scale;
  void* out;
  float* lse;
  int32_t num_splits;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  int32_t draft_block = 0;  // TiDAR: 0 = no mask inside the draft block
};

pa_status run_decode_impl(const CallArgs& a, cudaEvent_t ev_start, cudaEvent_t ev_split);

pa_status run_decode(const CallArgs& a) {
  cudaEvent_t ev_start = t_ev_start, ev_split = t_ev_split;
  t_ev_start = t_ev_split = nullptr;
  return run_decode_impl(a, ev_start, ev_split);
}

pa_status run_decode_impl(const CallArgs& a, cudaEvent_t ev_start, cudaEvent_t ev_split) {
  pa_status st = check_shape(a.shape, a.kind);
  if (st != PA_OK) return st;
  const pa_shape& s = *a.shape;
  if (!std::isfinite(a.scale) || a.num_splits < 0) return PA_ERR_INVALID_ARG;
  if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens || !a.out) return PA_ERR_INVALID_ARG;
  if (!aligned(a.q, 16) || !aligned(a.k_cache, 16) || !aligned(a.v_cache, 16) || !aligned(a.out, 16) ||
      !aligned(a.block_tables, 4) || !aligned(a.context_lens, 4) || (a.lse && !aligned(a.lse, 4)))
    return PA_ERR_INVALID_ARG;
  if (a.kind == Kind::kFp8 &&
      (!a.k_scale || !a.v_scale || !aligned(a.k_scale, 16) || !aligned(a.v_scale, 16)))
    return PA_ERR_INVALID_ARG;
  if (a.kind == Kind::kTidar &&
      (!a.k_scratch || !a.v_scratch || !aligned(a.k_scratch, 16) || !aligned(a.v_scratch, 16)))
    return PA_ERR_INVALID_ARG;
  if (s.batch == 0) return PA_OK;

  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;
  Plan plan;
  if ((st = make_plan(a.shape, a.kind, a.num_splits, d, &plan)) != PA_OK) return st;
  if (plan.ws_bytes) {
    if (!a.workspace || a.workspace_bytes < plan.ws_bytes || !aligned(a.workspace, 256)) return PA_ERR_WORKSPACE;
  }

  const int B = s.batch, T = s.q_tokens, Hq = s.num_q_heads, Hkv = s.num_kv_heads, D = s.head_dim;
  const int P = s.page_size, G = Hq / Hkv;
  const bool fp8 = a.kind == Kind::kFp8;
  const uint64_t e = fp8 ? 1 : 2;

  static_assert(sizeof(SplitParams) % 64 == 0, "params must keep the descriptors aligned");
  SplitParams p;
  std::memset(&p, 0, sizeof(p));
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)T, (uint64_t)B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)T * Hq * D * 2};
    const uint32_t box[4] = {64u, (uint32_t)G, (uint32_t)T, 1u};
    const CUtensorMapDataType qt =
        a.kind == Kind::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_map(&p.tm_q, qt, a.q, dims, str, box)) return PA_ERR_INVALID_ARG;
  }
  // KV caches as 5-D (128-byte column chunk, slot, kv head, chunk index,
  // page): one box copies every chunk of BR rows of one page for the H2
  // heads of a unit, landing in shared memory as [chunk][head][row][128 B]
  // (or, for the query-row kernel, one chunk per box: [head][row][128 B]).
  const Geom& geo = plan.geo;
  const uint64_t nch = (uint64_t)D * e / 128;
  const uint32_t box_ch = geo.chunk_boxes ? 1u : (uint32_t)nch;
  {
    const uint64_t dims[5] = {128 / e, (uint64_t)P, (uint64_t)Hkv, nch, (uint64_t)s.num_pages};
    const uint64_t str[4] = {(uint64_t)Hkv * D * e, (uint64_t)D * e, 128, (uint64_t)P * Hkv * D * e};
    const uint32_t box[5] = {(uint32_t)(128 / e), (uint32_t)geo.BR, (uint32_t)geo.H2, box_ch, 1u};
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : (a.kind == Kind::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    if (!make_map(&p.tm_k, dt, a.k_cache, dims, str, box)) return PA_ERR_INVALID_ARG;
    if (!make_map(&p.tm_v, dt, a.v_cache, dims, str, box)) return PA_ERR_INVALID_ARG;
  }
  if (a.kind == Kind::kTidar) {
    // Rows T..TP-1 of the box fall outside the tensor and read as zeros.
    const uint64_t dims[5] = {64, (uint64_t)T, (uint64_t)Hkv, nch, (uint64_t)B};
    const uint64_t str[4] = {(uint64_t)Hkv * D * 2, (uint64_t)D * 2, 128, (uint64_t)T * Hkv * D * 2};
    const uint32_t box[5] = {64u, (uint32_t)geo.TP, (uint32_t)geo.H2, box_ch, 1u};
    if (!make_map(&p.tm_ks, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k_scratch, dims, str, box) ||
        !make_map(&p.tm_vs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.v_scratch, dims, str, box))
      return PA_ERR_INVALID_ARG;
  }
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.err_flags = d->err_flags;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.M = geo.M;
  p.P = P;
  p.H2 = geo.H2;
  p.NHG = geo.NHG;
  p.GT = geo.GT;
  p.TS = geo.TS;
  p.ilv = geo.ilv;
  p.BR = geo.BR;
  p.lbr = geo.lbr;
  p.TP = geo.TP;
  p.max_blocks = s.max_blocks_per_seq;
  p.num_pages = s.num_pages;
  p.num_splits = plan.balanced ? 0 : plan.splits;
  p.tidar = a.kind == Kind::kTidar ? 1 : 0;
  p.draft_block = a.draft_block > 0 && a.draft_block < T ? a.draft_block : T;
  p.grid = plan.grid;
  p.item_w = plan.balanced ? plan.item_w : 0;
  p.scale_log2 = (float)((double)a.scale * 1.4426950408889634);
  if (plan.ws_bytes) {
    p.part_o = static_cast<float*>(a.workspace);
    p.part_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + plan.part_lse_off);
  }
  // Fused combine: warp-level kernel, balanced schedule; the counters start
  // at zero (one memset per call; the kernel leaves them zero as well).
  const bool fused = plan.balanced && geo.path == kPathWarp && geo.k.fused &&
                     g_combine_mode.load(std::memory_order_relaxed) == 1;
  if (fused) {
    p.unit_count = reinterpret_cast<unsigned*>(static_cast<char*>(a.workspace) + plan.count_off);
    if (cudaMemsetAsync(p.unit_count, 0, (size_t)B * geo.NHG * sizeof(unsigned), a.stream) != cudaSuccess)
      return PA_ERR_CUDA;
  }

  const SplitKernel k = geo.k;
  if ((st = ensure_kernel_ready(d, k)) != PA_OK) return st;
  const dim3 grid = plan.balanced ? dim3(plan.grid) : dim3(B * geo.NHG, plan.splits);
  void* args[] = {&p};
  if (ev_start && cudaEventRecord(ev_start, a.stream) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaLaunchKernel(k.fn, grid, dim3(k.threads), args, plan.smem, a.stream) != cudaSuccess)
    return PA_ERR_CUDA;
  if (ev_split && cudaEventRecord(ev_split, a.stream) != cudaSuccess) return PA_ERR_CUDA;

  if ((plan.balanced && !fused) || plan.splits > 1) {
    ReduceParams r;
    std::memset(&r, 0, sizeof(r));
    r.part_o = p.part_o;
    r.part_lse = p.part_lse;
    r.out = p.out;
    r.lse = p.lse;
    r.B = B;
    r.T = T;
    r.Hq = Hq;
    r.D = D;
    r.context_lens = p.context_lens;
    r.G = G;
    r.M = geo.M;
    r.H2 = geo.H2;
    r.NHG = geo.NHG;
    r.GT = geo.GT;
    r.P = P;
    r.max_blocks = s.max_blocks_per_seq;
    r.tidar = p.tidar;
    r.item_w = p.item_w;
    r.num_splits = plan.balanced ? 0 : plan.splits;
    r.out_f16 = a.kind == Kind::kF16 ? 1 : 0;
    r.grid = plan.grid;
    // Programmatic dependent launch: the reduce grid may start while the
    // split grid drains and waits (griddepcontrol.wait) for its results.
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    if (plan.balanced) {
      cfg.gridDim = dim3(B * geo.NHG, (geo.M + 3) / 4);
      err = cudaLaunchKernelEx(&cfg, pa::pa_reduce_balanced_kernel, r);
    } else {
      cfg.gridDim = dim3((unsigned)(((size_t)B * T * Hq + 3) / 4));
      err = cudaLaunchKernelEx(&cfg, pa::pa_reduce_splits_kernel, r);
    }
    if (err != cudaSuccess) return PA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t pa_decode_workspace_size(const pa_shape* shape, int32_t num_splits) {
  if (check_shape(shape, Kind::kBf16) != PA_OK && check_shape(shape, Kind::kFp8) != PA_OK) return 0;
  if (num_splits < 0) return 0;
  if (num_splits == 1) return 0;
  if (num_splits > 1) {
    const size_t rows = (size_t)shape->batch * shape->q_tokens * shape->num_q_heads * num_splits;
    return align256(rows * shape->head_dim * sizeof(float)) + align256(rows * sizeof(float));
  }
  DeviceState* d = nullptr;
  if (device_state(&d) != PA_OK) return 0;
  // The balanced plan depends on the kind and the kernel (through the
  // instance's fixed shared memory, its rows per unit and the draft block's
  // extra page); take the largest plan over every decode entry point and
  // every kernel selection, so that the size holds whatever
  // pa_decode_set_kernel_path chooses.
  size_t best = 0;
  for (Kind kind : {Kind::kBf16, Kind::kF16, Kind::kFp8, Kind::kTidar}) {
    if (check_shape(shape, kind) != PA_OK) continue;
    for (int path : {kPathWarp, kPathUmma, kPathQrow, kPathPair}) {
      Plan plan;
      if (make_plan(shape, kind, 0, d, &plan, path) == PA_OK && plan.ws_bytes > best) best = plan.ws_bytes;
    }
  }
  return best;
}

int32_t pa_decode_choose_splits(const pa_shape* shape, int32_t fp8_kv) {
  const Kind kind = fp8_kv ? Kind::kFp8 : Kind::kBf16;
  if (check_shape(shape, kind) != PA_OK) return -1;
  DeviceState* d = nullptr;
  if (device_state(&d) != PA_OK) return -1;
  Plan plan;
  if (make_plan(shape, kind, 0, d, &plan) != PA_OK) return -1;
  return plan.balanced ? 0 : plan.splits;
}

pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                    const int32_t* context_lens, const pa_shape* shape, float scale, void* out, float* lse,
                    int32_t num_splits, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  CallArgs a{Kind::kBf16, q, k_cache, v_cache, nullptr, nullptr, nullptr, nullptr, block_tables, context_lens,
             shape, scale, out, lse, num_splits, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)};
  return run_decode(a);
}

pa_status pa_decode_fp8(const void* q, const uint8_t* k_cache, const uint8_t* v_cache, const float* k_scale,
                        const float* v_scale, const int32_t* block_tables, const int32_t* context_lens,
                        const pa_shape* shape, float scale, void* out, float* lse, int32_t num_splits,
                        void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  CallArgs a{Kind::kFp8, q, k_cache, v_cache, k_scale, v_scale, nullptr, nullptr, block_tables, context_lens,
             shape, scale, out, lse, num_splits, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)};
  return run_decode(a);
}

pa_status pa_decode_tidar(const void* q, const void* k_cache, const void* v_cache, const void* k_scratch,
                          const void* v_scratch, const int32_t* block_tables, const int32_t* context_lens,
                          const pa_shape* shape, float scale, void* out, float* lse, int32_t num_splits,
                          void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  CallArgs a{Kind::kTidar, q, k_cache, v_cache, nullptr, nullptr, k_scratch, v_scratch, block_tables,
             context_lens, shape, scale, out, lse, num_splits, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream)};
  return run_decode(a);
}

pa_status pa_decode_f16(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        const int32_t* context_lens, const pa_shape* shape, float scale, void* out, float* lse,
                        int32_t num_splits, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  CallArgs a{Kind::kF16, q, k_cache, v_cache, nullptr, nullptr, nullptr, nullptr, block_tables, context_lens,
             shape, scale, out, lse, num_splits, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)};
  return run_decode(a);
}

pa_status pa_decode_tidar_masked(const void* q, const void* k_cache, const void* v_cache, const void* k_scratch,
                                 const void* v_scratch, const int32_t* block_tables, const int32_t* context_lens,
                                 const pa_shape* shape, float scale, int32_t draft_block, void* out, float* lse,
                                 int32_t num_splits, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (draft_block < 1) return PA_ERR_INVALID_ARG;
  CallArgs a{Kind::kTidar, q, k_cache, v_cache, nullptr, nullptr, k_scratch, v_scratch, block_tables,
             context_lens, shape, scale, out, lse, num_splits, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), draft_block};
  return run_decode(a);
}

}  // extern "C"

namespace {

pa_status run_reduce(const float* part_out, const float* part_lse, int32_t num_splits, const pa_shape* shape,
                     void* out, float* lse, pa_stream_t stream, bool out_f16) {
  if (!shape || !part_out || !part_lse || !out || num_splits < 1) return PA_ERR_INVALID_ARG;
  if (shape->batch < 0 || shape->q_tokens < 1 || shape->num_q_heads < 1 || shape->head_dim < 4 ||
      shape->head_dim % 4 || shape->head_dim > 1024)
    return PA_ERR_INVALID_ARG;
  if (!aligned(part_out, 16) || !aligned(part_lse, 4) || !aligned(out, 8) || (lse && !aligned(lse, 4)))
    return PA_ERR_INVALID_ARG;
  if (shape->batch == 0) return PA_OK;
  ReduceParams r;
  std::memset(&r, 0, sizeof(r));
  r.part_o = part_out;
  r.part_lse = part_lse;
  r.out = static_cast<__nv_bfloat16*>(out);
  r.lse = lse;
  r.B = shape->batch;
  r.T = shape->q_tokens;
  r.Hq = shape->num_q_heads;
  r.D = shape->head_dim;
  r.num_splits = num_splits;
  r.out_f16 = out_f16 ? 1 : 0;
  const size_t rows = (size_t)r.B * r.T * r.Hq;
  void* rargs[] = {&r};
  if (cudaLaunchKernel(reinterpret_cast<const void*>(&pa::pa_reduce_splits_kernel), dim3((unsigned)((rows + 3) / 4)),
                       dim3(128), rargs, 0, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

pa_status pa_decode_reduce(const float* part_out, const float* part_lse, int32_t num_splits, const pa_shape* shape,
                           void* out, float* lse, pa_stream_t stream) {
  return run_reduce(part_out, part_lse, num_splits, shape, out, lse, stream, false);
}

pa_status pa_decode_reduce_f16(const float* part_out, const float* part_lse, int32_t num_splits,
                               const pa_shape* shape, void* out, float* lse, pa_stream_t stream) {
  return run_reduce(part_out, part_lse, num_splits, shape, out, lse, stream, true);
}

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape or format";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

// Split-K scratch for pa_decode_noalloc: reserved statically in every
// device's copy of this module, so the entry point never allocates.
static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

static void* g_noalloc_ptr[kMaxDevices];
static std::atomic<bool> g_noalloc_ready[kMaxDevices];  // publishes g_noalloc_ptr (release/acquire)

// Device address of this device's scratch array. In host code the array's
// name stands for a host-side shadow, so the address must come from the
// runtime; looked up once per device, with that device current.
static pa_status noalloc_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  if (!g_noalloc_ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_noalloc_ready[dev].load(std::memory_order_relaxed)) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_pa_noalloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
      g_noalloc_ptr[dev] = p;
      g_noalloc_ready[dev].store(true, std::memory_order_release);
    }
  }
  *ptr = g_noalloc_ptr[dev];
  return PA_OK;
}

pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, const pa_shape* shape, float scale, void* out,
                            float* lse, int32_t num_splits, pa_stream_t stream) {
  pa_status st = check_shape(shape, Kind::kBf16);
  if (st != PA_OK) return st;
  if (num_splits < 0) return PA_ERR_INVALID_ARG;
  size_t need = 0;
  if (shape->batch > 0) {
    DeviceState* d = nullptr;
    if ((st = device_state(&d)) != PA_OK) return st;
    Plan plan;
    if ((st = make_plan(shape, Kind::kBf16, num_splits, d, &plan)) != PA_OK) return st;
    need = plan.ws_bytes;
  }
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0 && (st = noalloc_scratch(&ws)) != PA_OK) return st;
  return pa_decode(q, k_cache, v_cache, block_tables, context_lens, shape, scale, out, lse, num_splits, ws, need,
                   stream);
}

pa_status pa_decode_set_combine(int32_t mode) {
  if (mode < 0 || mode > 1) return PA_ERR_INVALID_ARG;
  g_combine_mode.store(mode, std::memory_order_relaxed);
  return PA_OK;
}

pa_status pa_decode_set_kernel_path(int32_t path) {
  if (path < kPathAuto || path > kPathPair) return PA_ERR_INVALID_ARG;
  g_kernel_path.store(path, std::memory_order_relaxed);
  return PA_OK;
}

int32_t pa_decode_kernel_for(const pa_shape* shape, int32_t format) {
  if (format < 0 || format > 3) return -1;
  const Kind kind = format == 1 ? Kind::kFp8 : format == 2 ? Kind::kF16 : format == 3 ? Kind::kTidar : Kind::kBf16;
  if (check_shape(shape, kind) != PA_OK) return -1;
  Geom g;
  if (pick_geometry(shape, kind, &g) != PA_OK) return -1;
  return g.path;
}

int32_t pa_decode_heads_per_unit(const pa_shape* shape, int32_t format) {
  if (format < 0 || format > 3) return -1;
  const Kind kind = format == 1 ? Kind::kFp8 : format == 2 ? Kind::kF16 : format == 3 ? Kind::kTidar : Kind::kBf16;
  if (check_shape(shape, kind) != PA_OK) return -1;
  Geom g;
  if (pick_geometry(shape, kind, &g) != PA_OK) return -1;
  return g.H2;
}

pa_status pa_decode_profile_events(void* start_event, void* split_done_event) {
  t_ev_start = static_cast<cudaEvent_t>(start_event);
  t_ev_split = static_cast<cudaEvent_t>(split_done_event);
  return PA_OK;
}

pa_status pa_decode_device_error(int32_t* flags) {
  if (!flags) return PA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  pa_status st = device_state(&d);
  if (st != PA_OK) return st;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_pa_err_flags, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_pa_err_flags, &zero, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
  *flags = v;
  return PA_OK;
}

}  // extern "C"
