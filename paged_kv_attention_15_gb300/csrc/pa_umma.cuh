// Paged-KV decode attention on the fifth-generation tensor cores (tcgen05)
// for work units with many query rows per kv head: the fp8 KV cache, and
// draft blocks (TiDAR) of 16-bit caches.
//
// Token-major formulation. A work unit is (sequence, H2 kv heads) with
// N = H2 * G * T query rows. A pipeline stage holds 128 key rows: TSK =
// 128 / H2 tokens of each head, in row order kr = h * TSK + t. Per stage
//   S^T [128 key rows x N] = K_stage [128 x D] . Q^T      (M = 128, in TMEM)
//   softmax over the tokens, per query row (column), in base 2
//   O_h^T [D x G*T] += V_h^T [D x TSK] . P_h^T [TSK x G*T]  (per head h)
// Key row kr only pairs with the query rows of its own head: S^T holds the
// scores of every (key row, query row) pair, and a softmax thread reads
// only its head's columns; P^T and O^T are kept per head.
// Sources: ROCm blog "Implementing a High-Performance Custom Diffusion
// Attention Kernel with FlyDSL" (introduction items 1-3: paged KV caches,
// scratch storage for draft tokens, FlashAttention-style online softmax with
// split-K; "Match MFMA Operands to the Desired Fragment Layout": the
// probabilities feed the P x V product without a round trip through a
// transpose) and the MSLK pull request "[ROCm] Add FlyDSL paged-attention
// decode backend (dense + fp8) with benchmark" (Kernels: head-packed
// matrix-core decode, native fp8 e4m3fn KV with symmetric per-token scale,
// split-K partial combine).
//
// Roles of the 512 threads (one CTA per SM; four warpgroups, registers
// rebalanced between them with setmaxnreg):
//  - warps 0-3, softmax: warp w reads TMEM lanes 32w..32w+31 = key rows
//    (the tensor-memory quadrant rule), holds each row's online-softmax
//    state for its head's query rows (columns), writes P^T to shared memory,
//    rescales O^T in TMEM when a running max moves by more than the slack,
//    and writes the outputs.
//  - warps 4-7, K converters: turn a stage's K page boxes into the MMA's K
//    operand (fp8: e4m3fn -> f16, exact; 16-bit: a copy that puts the pages'
//    rows in token order), one key row per thread; fp8: they also read the
//    per-token K scales for the softmax, and convert Q to f16.
//  - warps 8-11, V converters: the same for V into the V^T operand (fp8:
//    the per-token V scale folded in); rows past the valid tokens are zero.
//  - warp 12, producer: block-table walk, one TMA box per page for K and V,
//    Q boxes per work item; publishes each stage's page ids.
//  - warp 13: allocates the tensor memory; lane 0 issues every tcgen05.mma
//    and commits their completion to mbarriers. Warps 14-15 idle.
// Every wait is bounded in time; on a timeout the CTA raises an abort flag
// and a device error bit, the roles finish without waiting, and the rows of
// the items cut short are written as NaN.
#pragma once

#include "pa_kernels.cuh"
#include "pa_tc.cuh"

namespace pa {

constexpr int kUThreads = 512;
constexpr int kUKConvWarp0 = 4;
constexpr int kUVConvWarp0 = 8;
constexpr int kUProducerWarp = 12;   // K pages, Q, page-id table
constexpr int kUMmaWarp = 13;
constexpr int kUVProducerWarp = 14;  // V pages
constexpr int kUPvWarp = 15;         // issues the P V products
constexpr int kSmemLimit = 232448;  // 227 KB of dynamic shared memory per CTA
// Registers per thread after the split (launched with 65536 / 512 = 128):
// softmax 200, converters 104, producer/MMA warpgroup 96;
// 200 * 128 + 104 * 256 + 96 * 128 = 64512 <= 65536.
constexpr int kRegSoftmax = 200, kRegConv = 104, kRegOther = 96;
constexpr int kULaunchRegs = 65536 / kUThreads;  // registers per thread at launch (the pool the split draws on)
static_assert(kRegSoftmax * 128 + kRegConv * 256 + kRegOther * 128 <= kUThreads * kULaunchRegs, "register split");

template <int D, int KV, int GT, int N>
struct UCfg {
  static constexpr bool FP8 = KV == kKvFp8;
  static constexpr bool BF16 = KV == kKvBf16;  // MMA operand type: bf16, else f16
  static constexpr int H2 = N / GT;            // kv heads per unit
  static constexpr int TSK = 128 / H2;         // tokens of each head per stage
  static constexpr int E = FP8 ? 1 : 2;        // bytes per cache element
  static constexpr int RCH = D * E / 128;      // 128-byte chunks per cache row
  static constexpr int RAWT = 128 * D * E;     // K (or V) bytes of a stage as copied
  static constexpr int RAW = 2 * RAWT;
  static constexpr int NRAW = 2;               // stages of page boxes in flight
  static constexpr int NKP = D / 64;           // K operand pieces per stage (64 columns, 16 KB)
  static constexpr int KPB = 16384;
  static constexpr int NKPS = 2;               // K piece slots
  static constexpr int NVT = D / 128;          // 128-column tiles of the V^T operand
  // V^T operand sub-tile: one 128-column tile of SUBR key rows of one head,
  // [2 chunks of 64 columns][SUBR rows][128 B]; a ring of two, so the V
  // converters fill one while the MMAs read the other.
  static constexpr int SUBR = TSK < 64 ? TSK : 64;
  static constexpr int NKH = TSK / SUBR;  // sub-tiles per head and tile
  static constexpr int SUBB = SUBR * 256;
  static constexpr int NVS = 2;
  static constexpr int VTB = NVS * SUBB;
  static constexpr int QB = N * D * 2;         // Q operand tile
  static constexpr int PSW = GT * 2;           // bytes of a P^T row (the swizzle width)
  static constexpr int PH = TSK * PSW;         // P^T bytes of one head
  static constexpr int PB = round_up(H2 * PH, 1024);
  static constexpr int OFF_KP = NRAW * RAW;
  static constexpr int OFF_VT = OFF_KP + NKPS * KPB;
  static constexpr int OFF_Q = OFF_VT + VTB;
  static constexpr int OFF_PT = OFF_Q + round_up(QB, 1024);
  static constexpr int REST = 1024 + 3 * 256 + 512 + 64 + 128 + (FP8 ? 4096 : 0);  // exchange arrays, barriers, ids, scales
  static constexpr int NPT = OFF_PT + 2 * PB + REST + 1024 + 1024 <= kSmemLimit ? 2 : 1;
  static constexpr int OFF_RED = OFF_PT + NPT * PB;  // [4 warps][64] floats
  static constexpr int OFF_ALPHA = OFF_RED + 1024;   // [N] floats
  static constexpr int OFF_COLL = OFF_ALPHA + 256;   // [N] floats
  static constexpr int OFF_COLM = OFF_COLL + 256;    // [N] floats
  static constexpr int OFF_BAR = OFF_COLM + 256;     // 64 mbarrier slots
  static constexpr int OFF_MISC = OFF_BAR + 512;     // tensor-memory base, abort flag
  static constexpr int OFF_IDS = OFF_MISC + 64;      // page ids of a stage: [4][8] ints
  // fp8 per-row scales of a stage, a ring of four stages: the K converters
  // can run two stages ahead of the softmax that reads them
  static constexpr int OFF_KSS = OFF_IDS + 128;      // fp8: scale_log2 * K scale per key row: [4][128] floats
  static constexpr int OFF_VSS = OFF_KSS + (FP8 ? 2048 : 0);  // fp8: V scale per key row: [4][128] floats
  static constexpr int OFF_TABLE = OFF_VSS + (FP8 ? 2048 : 0);  // balanced mode: per-sequence lengths, starts
  static constexpr int SMEM_FIXED = OFF_TABLE + 1024;  // + 1024 to align the dynamic base
  // tensor-memory columns: S^T [2][N], then O^T [2 items][NVT][N]
  static constexpr int TM_O = 2 * N;
  static constexpr int TM_USED = 2 * N + 2 * NVT * N;
  static constexpr int TM_COLS = TM_USED <= 32 ? 32 : TM_USED <= 64 ? 64 : TM_USED <= 128 ? 128 : TM_USED <= 256 ? 256 : 512;
  static constexpr uint32_t PSWZ = PSW == 32 ? kSwz32 : (PSW == 64 ? kSwz64 : kSwz128);
  static constexpr int PSHIFT = PSW == 32 ? 2 : (PSW == 64 ? 1 : 0);  // P^T swizzle: unit ^ ((row & 7) >> PSHIFT)
  static_assert(D == 128 || (FP8 && D == 256), "unsupported head_dim");
  static_assert(GT == 16 || GT == 32 || GT == 64, "unsupported query rows per kv head");
  static_assert(H2 == 1 || H2 == 2 || H2 == 4, "unsupported heads per unit");
  static_assert(N <= 64, "unsupported rows per unit");
  // whether this instance's tiles fit the SM (checked again by the kernel)
  static constexpr bool FITS = SMEM_FIXED + 1024 <= kSmemLimit && TM_USED <= 512;
};

// Barrier slots (8 bytes each) inside OFF_BAR.
enum UBar {
  kBRawKFull = 0,   // [2] K page boxes of a stage landed (tx bytes)
  kBRawKEmpty = 2,  // [2] converters done with them (4 warps)
  kBRawVFull = 4,   // [2] V page boxes landed (tx bytes)
  kBRawVEmpty = 6,  // [2] converters done with them (4 warps)
  kBKpFull = 8,     // [2] K piece written (4 warps)
  kBKpEmpty = 10,   // [2] K piece read by its MMAs (commit)
  kBVtFull = 12,    // [2] V sub-tile written (4 warps)
  kBVtEmpty = 32,   // [2] V sub-tile read (commit)
  kBSFull = 14,     // [2] S^T computed (commit)
  kBSEmpty = 16,    // [2] S^T read by the softmax (4 warps)
  kBPFull = 18,     // [2] P^T written (4 warps)
  kBPEmpty = 20,    // [2] P^T read and O^T updated (commit)
  kBOFull = 22,     // [2] an item's O^T complete (commit)
  kBOEmpty = 24,    // [2] an item's O^T read by the epilogue (4 warps)
  kBQFull = 26,     // Q landed (tx bytes)
  kBQReady = 27,    // fp8: Q converted to f16 (4 warps)
  kBQEmpty = 28,    // Q no longer read (commit)
  kBDone = 29,      // every MMA of the CTA complete (a commit by each issuer)
  kBKssFull = 34,   // [4] fp8: a stage's K and V scales written (4 warps)
  kBCount = 38
};

// Max or sum of GT values over the 32 lanes of a warp, by halving exchange:
// after it, lane l holds the reduction of columns col0(l) .. col0(l)+R-1
// (R = max(1, GT / 32)) in v[0..R-1], where col0 = (l >> 1) for GT = 16,
// l for GT = 32 and 2 l for GT = 64.
template <int GT, bool MAX>
__device__ __forceinline__ void warp_columns_reduce(float* v, int lane) {
  int n = GT;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool up = lane & o;
#pragma unroll
      for (int i = 0; i < GT / 2; ++i) {
        if (i < n / 2) {
          const float send = up ? v[i] : v[i + n / 2];
          const float keep = up ? v[i + n / 2] : v[i];
          const float recv = __shfl_xor_sync(0xffffffffu, send, o);
          v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
      }
      n >>= 1;
    } else {
      const float recv = __shfl_xor_sync(0xffffffffu, v[0], o);
      v[0] = MAX ? fmaxf(v[0], recv) : v[0] + recv;
    }
  }
}

template <int GT>
__device__ __forceinline__ int reduced_col0(int lane) {
  return GT == 16 ? (lane >> 1) : (GT == 32 ? lane : 2 * lane);
}

// Maximum of x over the 32 lanes of the warp, in every lane.
__device__ __forceinline__ float redux_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}


template <int D, int KV, int GT, int N>
__global__ void __launch_bounds__(kUThreads, 1) pa_umma_kernel(const __grid_constant__ SplitParams p) {
  using C = UCfg<D, KV, GT, N>;
  static_assert(C::FITS, "shared or tensor memory");
  constexpr bool FP8 = C::FP8;
  constexpr int H2 = C::H2;
  constexpr int TSK = C::TSK;
  constexpr int NVT = C::NVT;
  constexpr int NPT = C::NPT;
  extern __shared__ uint8_t smem_raw[];
  // (pointer arithmetic on the shared array, so that accesses through smem
  // stay shared-memory accesses)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  // 16-byte shared loads and stores by shared address, as ordinary C++
  // accesses (the compiler may overlap them; mbarrier waits order them)
  auto lds = [&](uint32_t a) { return *reinterpret_cast<const uint4*>(smem + (a - sbase)); };
  auto sts = [&](uint32_t a, uint4 v) { *reinterpret_cast<uint4*>(smem + (a - sbase)) = v; };
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  int* s_ctx = reinterpret_cast<int*>(smem + C::OFF_TABLE);
  int* s_start = s_ctx + (p.num_splits == 0 ? p.B : 0);
  const float NEG_INF = -__int_as_float(0x7f800000);

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBRawKFull + s), 1);
      mbar_init(bar(kBRawKEmpty + s), 4);
      mbar_init(bar(kBRawVFull + s), 1);
      mbar_init(bar(kBRawVEmpty + s), 4);
      mbar_init(bar(kBKpFull + s), 4);
      mbar_init(bar(kBKpEmpty + s), 1);
      mbar_init(bar(kBSFull + s), 1);
      mbar_init(bar(kBSEmpty + s), 4);
      mbar_init(bar(kBPFull + s), 4);
      mbar_init(bar(kBPEmpty + s), 1);
      mbar_init(bar(kBOFull + s), 1);
      mbar_init(bar(kBOEmpty + s), 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBVtFull + s), 4);
      mbar_init(bar(kBVtEmpty + s), 1);
    }
    mbar_init(bar(kBQFull), 1);
    mbar_init(bar(kBQReady), 4);
    mbar_init(bar(kBQEmpty), 1);
    mbar_init(bar(kBDone), 2);
    for (int s = 0; s < 4; ++s) mbar_init(bar(kBKssFull + s), 4);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kUMmaWarp) tmem_alloc(sbase + C::OFF_MISC, C::TM_COLS);
  if (p.num_splits == 0) {
    for (int i = tid; i < p.B; i += kUThreads) s_ctx[i] = clamp_ctx(p, __ldg(p.context_lens + i));
    __syncthreads();
    if (warp == 0) {  // exclusive prefix sum of virtual pages per sequence
      int carry = 0;
      if (lane == 0) s_start[0] = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int i = base + lane;
        int v = i < p.B ? unit_vpages(s_ctx[i], p.P, p.tidar, p.item_w) : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += n;
        }
        if (i < p.B) s_start[i + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *s_tmem;

  const int P = p.P;
  const int lp = 31 - __clz(P);  // log2 of the page size (a power of two)
  // Raw stage layout: [page box][chunk][head][box row][128 B]; a box holds
  // BR rows of the H2 heads (scratch stage: TP rows).
  const uint32_t box_bytes = (uint32_t)(C::RCH * H2 * p.BR * 128);
  const uint32_t cstride = (uint32_t)(H2 * p.BR * 128);
  const uint32_t scr_cstride = (uint32_t)(H2 * p.TP * 128);
  Cursor cur;
  cursor_init(p, s_start, cur);
  Item it;
  bool ok = true;

  const int wg = warp >> 2;  // warpgroup: 0 softmax, 1 K converters, 2 V converters, 3 producer + MMA
  int* s_ids = reinterpret_cast<int*>(smem + C::OFF_IDS);  // [st & 3][8]: page ids of stage st

  if (wg == 3) {
   regs_dec<kRegOther>();
   if (warp == kUProducerWarp || warp == kUVProducerWarp) {
    // ================================================================ producers
    // Two warps: one copies the K pages (and Q, and publishes the page
    // ids), the other the V pages, so that neither waits behind the other's
    // ring (V slots are released later than K slots).
    const int kv = warp == kUVProducerWarp ? 1 : 0;
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    if (lane == 0) {
      if (kv == 0) prefetch_tensormap(&p.tm_q);
      prefetch_tensormap(kv ? &p.tm_v : &p.tm_k);
    }
    int stage = 0, qn = 0;
    uint32_t filled = 0, fill_parity = 0;
    const uint32_t row_bytes = (uint32_t)(H2 * D * C::E);
    while (ok && next_item(p, s_ctx, s_start, cur, it)) {
      if (it.nst == 0) continue;
      if (kv == 0 && qn >= 1)
        ok = __all_sync(0xffffffffu, mbar_wait_sleep(bar(kBQEmpty), (qn - 1) & 1, kWaitLimitNs, s_abort));
      if (!ok) break;
      if (kv == 0 && lane == 0) {
        const uint32_t qdst = sbase + C::OFF_Q;
        mbar_arrive_expect_tx(bar(kBQFull), C::QB);
        for (int hl = 0; hl < H2; ++hl)
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(qdst + c * (N * 128) + hl * GT * 128, &p.tm_q, bar(kBQFull), c * 64,
                        (it.hg * H2 + hl) * p.G, 0, it.b, pol_q);
      }
      ++qn;
      const int32_t* bt_row = p.block_tables + (size_t)it.b * p.max_blocks;
      const int pbase = it.tok0 / P;
      const int npages = it.tok_end > it.tok0 ? (it.tok_end - 1) / P + 1 - pbase : 0;
      int ibase = 0;
      int ids = lane < npages ? __ldg(bt_row + pbase + lane) : 0;
      int ids_next = 32 + lane < npages ? __ldg(bt_row + pbase + 32 + lane) : 0;
      for (int j = 0; j < it.nst; ++j, ++stage) {
        const int slot = stage & 1;
        const bool scr = it.scratch && j == it.nst - 1;
        const int t_first = it.tok0 + j * TSK;
        const int valid = scr ? 0 : min(TSK, it.tok_end - t_first);
        const int pidx0 = scr ? 0 : t_first / P - pbase;
        while (!scr && pidx0 >= ibase + 32) {
          ibase += 32;
          ids = ids_next;
          ids_next = ibase + 32 + lane < npages ? __ldg(bt_row + pbase + ibase + 32 + lane) : 0;
        }
        const int npg = scr ? 0 : (P < TSK ? (valid + P - 1) / P : 1);
        filled |= 1u << slot;
        fill_parity = (fill_parity & ~(1u << slot)) | (uint32_t((stage >> 1) & 1) << slot);
        {
          if (stage >= 2) {
            ok = __all_sync(0xffffffffu, mbar_wait_sleep(bar((kv ? kBRawVEmpty : kBRawKEmpty) + slot),
                                                   ((stage >> 1) - 1) & 1, kWaitLimitNs, s_abort));
            if (!ok) break;
          }
          if (kv == 0) {
            // the stage's page ids for the converters (read after the K or V
            // boxes land; the ring of four outlives both raw slots)
            const int pid = __shfl_sync(0xffffffffu, ids, (pidx0 - ibase + (lane & 7)) & 31);
            if (lane < npg) s_ids[(stage & 3) * 8 + lane] = pid;
            __syncwarp();
          }
          const uint32_t full = bar((kv ? kBRawVFull : kBRawKFull) + slot);
          const uint32_t dst = sbase + slot * C::RAW + kv * C::RAWT;
          const CUtensorMap* map = kv ? &p.tm_v : &p.tm_k;
          if (scr) {
            if (lane == 0) {  // rows T..TP-1 of the box lie outside the tensor: zero filled
              mbar_arrive_expect_tx(full, C::RCH * H2 * p.TP * 128);
              tma_load_5d(dst, kv ? &p.tm_vs : &p.tm_ks, full, 0, 0, it.hg * H2, 0, it.b, pol_kv);
            }
          } else if (P < TSK) {  // whole pages, one box each
            if (lane == 0) mbar_arrive_expect_tx(full, npg * P * row_bytes);
            for (int i = 0; i < npg; ++i) {
              const int page = __shfl_sync(0xffffffffu, ids, pidx0 - ibase + i);
              if (lane == 0) tma_load_5d(dst + i * box_bytes, map, full, 0, 0, it.hg * H2, 0, page, pol_kv);
            }
          } else {  // TSK rows of one page
            const int row0 = t_first & (P - 1);
            const int page = __shfl_sync(0xffffffffu, ids, pidx0 - ibase);
            if (lane == 0) {
              mbar_arrive_expect_tx(full, TSK * row_bytes);
              tma_load_5d(dst, map, full, 0, row0, it.hg * H2, 0, page, pol_kv);
            }
          }
        }
        if (!ok) break;
      }
    }
    launch_dependents();
    if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
    {  // let every copy this warp issued land before the CTA can exit
      const int zero = 0;
      const volatile int* no_abort = &zero;
      for (int s2 = 0; s2 < 2; ++s2)
        if (filled >> s2 & 1)
          mbar_wait(bar((kv ? kBRawVFull : kBRawKFull) + s2), fill_parity >> s2 & 1, kWaitLimitNs, no_abort);
      if (kv == 0 && qn > 0) mbar_wait(bar(kBQFull), (qn - 1) & 1, kWaitLimitNs, no_abort);
    }
   } else if (warp == kUMmaWarp || warp == kUPvWarp) {
    // ================================================================ MMA issuers
    // Two threads issue the MMAs, one per product, so that neither waits
    // behind the other's operands: lane 0 of warp 13 computes S^T = K Q^T
    // stage by stage, lane 0 of warp 15 the P V products. They write
    // different tensor-memory columns and meet only through the softmax
    // (S -> P, and the rescale of O). Each shares its SM sub-partition with
    // busy warps, so an MMA is one add to a precomputed descriptor and the
    // loops over pieces, k-steps, heads and tiles are unrolled. tcgen05
    // fences follow only the waits that hand tensor memory between threads
    // (the S and O buffers); operands in shared memory are ordered by the
    // writers' proxy fences and the mbarriers.
    if (lane == 0) {
      constexpr bool BF = C::BF16;
      int st = 0, qn = 0, oi = 0;
      if (warp == kUMmaWarp) {
        constexpr uint32_t idS = idesc_f16(128, N, BF, false, false);
        const uint64_t dK0 = smem_desc(sbase + C::OFF_KP, 16, 1024, kSwz128);
        const uint64_t dQ0 = smem_desc(sbase + C::OFF_Q, 16, 1024, kSwz128);
        int kpi = 0;
        while (next_item(p, s_ctx, s_start, cur, it)) {
          if (it.nst == 0) continue;
          if (ok) {
            ok = mbar_wait_sleep(bar(FP8 ? kBQReady : kBQFull), qn & 1, kWaitLimitNs, s_abort);
            if (!ok) raise_abort(s_abort, p.err_flags);
          }
          ++qn;
          for (int j = 0; j < it.nst; ++j, ++st) {
            const int sb = st & 1;
            if (ok && st >= 2) {
              ok = mbar_wait_sleep(bar(kBSEmpty + sb), ((st >> 1) - 1) & 1, kWaitLimitNs, s_abort);
              if (!ok) raise_abort(s_abort, p.err_flags);
            }
            tc_fence_after();
            const uint32_t d_s = tm + (uint32_t)(sb * N);
#pragma unroll
            for (int c = 0; c < C::NKP; ++c, ++kpi) {
              const int ks = kpi & 1;
              if (ok) {
                ok = mbar_wait_sleep(bar(kBKpFull + ks), (kpi >> 1) & 1, kWaitLimitNs, s_abort);
                if (!ok) raise_abort(s_abort, p.err_flags);
              }
              if (ok) {
                const uint64_t dK = dK0 + (uint64_t)(ks * (C::KPB >> 4));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  umma_f16(d_s, dK + 2 * k, dQ0 + (uint64_t)(((c * N * 128) >> 4) + 2 * k), idS,
                           (c | k) ? 1u : 0u);
              }
              umma_commit(bar(kBKpEmpty + ks));
            }
            umma_commit(bar(kBSFull + sb));
            if (j == it.nst - 1) umma_commit(bar(kBQEmpty));
          }
        }
      } else {
        constexpr uint32_t idPV = idesc_f16(128, GT, BF, true, true);
        const uint64_t dV0 = smem_desc(sbase + C::OFF_VT, C::SUBR * 128, 1024, kSwz128);
        const uint64_t dP0 = smem_desc(sbase + C::OFF_PT, C::PH, 8 * C::PSW, C::PSWZ);
        int vti = 0;
        while (next_item(p, s_ctx, s_start, cur, it)) {
          if (it.nst == 0) continue;
          const int ob = oi & 1;
          for (int j = 0; j < it.nst; ++j, ++st) {
            if (ok && j == 0 && oi >= 2) {  // the epilogue of item oi - 2 has read this O buffer
              ok = mbar_wait_sleep(bar(kBOEmpty + ob), ((oi >> 1) - 1) & 1, kWaitLimitNs, s_abort);
              if (!ok) raise_abort(s_abort, p.err_flags);
            }
            const int pb = st % NPT;
            if (ok) {
              ok = mbar_wait_sleep(bar(kBPFull + pb), (st / NPT) & 1, kWaitLimitNs, s_abort);
              if (!ok) raise_abort(s_abort, p.err_flags);
            }
            tc_fence_after();
            const uint64_t dP = dP0 + (uint64_t)((pb * C::PB) >> 4);
            const uint32_t acc0 = j == 0 ? 0u : 1u;
#pragma unroll
            for (int tt = 0; tt < NVT; ++tt) {
#pragma unroll
              for (int hk = 0; hk < H2 * C::NKH; ++hk, ++vti) {
                const int h = hk / C::NKH, kh = hk % C::NKH;
                const int vsl = vti & 1;
                if (ok) {
                  ok = mbar_wait_sleep(bar(kBVtFull + vsl), (vti >> 1) & 1, kWaitLimitNs, s_abort);
                  if (!ok) raise_abort(s_abort, p.err_flags);
                }
                if (ok) {
                  const uint32_t d_tm = tm + C::TM_O + (uint32_t)((ob * NVT + tt) * N + h * GT);
                  const uint64_t dV = dV0 + (uint64_t)((vsl * C::SUBB) >> 4);
#pragma unroll
                  for (int ks = 0; ks < C::SUBR / 16; ++ks)
                    umma_f16(d_tm, dV + (uint64_t)((ks * 16 * 128) >> 4),
                             dP + (uint64_t)((h * C::PH + (kh * C::SUBR + ks * 16) * C::PSW) >> 4), idPV,
                             (kh == 0 && ks == 0) ? acc0 : 1u);
                }
                umma_commit(bar(kBVtEmpty + vsl));
              }
            }
            umma_commit(bar(kBPEmpty + pb));
            if (j == it.nst - 1) umma_commit(bar(kBOFull + ob));
          }
          ++oi;
        }
      }
      // every MMA of this thread complete before the tensor memory is released
      umma_commit(bar(kBDone));
      if (warp == kUMmaWarp) {
        const int zero = 0;
        const volatile int* no_abort = &zero;
        mbar_wait(bar(kBDone), 0, kWaitLimitNs, no_abort);
      }
    }
    __syncwarp();
   }
  } else if (wg == 1 || wg == 2) {
    regs_dec<kRegConv>();
    // ================================================================ converters
    // Warpgroup 1 converts K (into the two K piece slots), warpgroup 2 V
    // (into the V tile slot); they run independently of each other.
    const bool isK = wg == 1;
    const int kr = tid - (isK ? 32 * kUKConvWarp0 : 32 * kUVConvWarp0);  // key row of this thread
    const int h = kr / TSK, t = kr % TSK;
    const int sw = t & 7;  // 128-byte swizzle phase of the row (raw and operand tiles)
    int stage = 0, qn = 0, kpi = 0, vti = 0;
    const uint32_t kp0 = sbase + C::OFF_KP, vt0 = sbase + C::OFF_VT;
    float* s_kss = reinterpret_cast<float*>(smem + C::OFF_KSS);
    float* s_vss = reinterpret_cast<float*>(smem + C::OFF_VSS);
    const float sl = p.scale_log2;
    while (next_item(p, s_ctx, s_start, cur, it)) {
      if (it.nst == 0) continue;
      const int g = it.hg * H2 + h;
      if (FP8 && isK) {  // Q: bf16 as copied -> f16 in place (the MMA takes both operands in f16)
        if (ok) {
          ok = mbar_wait_sleep(bar(kBQFull), qn & 1, kWaitLimitNs, s_abort);
          if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
        }
        if (ok) {
          uint4* q4 = reinterpret_cast<uint4*>(smem + C::OFF_Q);
          for (int i = kr; i < C::QB / 16; i += 128) {
            uint4 v = q4[i];
            v.x = bf16x2_to_f16x2(v.x);
            v.y = bf16x2_to_f16x2(v.y);
            v.z = bf16x2_to_f16x2(v.z);
            v.w = bf16x2_to_f16x2(v.w);
            q4[i] = v;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBQReady));
      }
      ++qn;
      for (int j = 0; j < it.nst; ++j) {
        const int st = stage + j, slot = st & 1;
        const bool scr = it.scratch && j == it.nst - 1;
        const int t_first = it.tok0 + j * TSK;
        const int valid = scr ? p.T : min(TSK, it.tok_end - t_first);
        // this row in the stage's boxes
        const bool has_src = scr ? t < p.TP : t < valid;
        const bool in_ctx = scr ? t < p.T : t < valid;
        const uint32_t roff = scr ? (uint32_t)(h * p.TP * 128 + t * 128)
                                  : (uint32_t)((t >> p.lbr) * box_bytes + h * p.BR * 128 + (t & (p.BR - 1)) * 128);
        const uint32_t cs = scr ? scr_cstride : cstride;
        if (ok) {
          ok = mbar_wait_sleep(bar((isK ? kBRawKFull : kBRawVFull) + slot), (st >> 1) & 1, kWaitLimitNs, s_abort);
          if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
        }
        // fp8, K converters: this token's K and V scales (its page id from
        // the producer's table); loaded now, published after the K pieces
        float ksc = 0.f, vsc_f = 0.f;
        if (FP8 && isK && ok && in_ctx) {
          const int tok = t_first + t;
          int pg = s_ids[(st & 3) * 8 + (P < TSK ? (t >> lp) : 0)];
          pg = (unsigned)pg < (unsigned)p.num_pages ? pg : 0;  // outside the pool: page 0's (finite) scales
          const size_t off = ((size_t)pg * P + (tok & (P - 1))) * p.Hkv + g;
          ksc = __ldg(p.k_scale + off);
          vsc_f = __ldg(p.v_scale + off);
        }
        const uint32_t rbase = sbase + slot * C::RAW + (isK ? 0 : C::RAWT);
        if (isK) {
          for (int c = 0; c < C::NKP; ++c, ++kpi) {
            const int ks = kpi & 1;
            if (ok && kpi >= 2) {
              ok = mbar_wait_sleep(bar(kBKpEmpty + ks), ((kpi >> 1) - 1) & 1, kWaitLimitNs, s_abort);
              if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
            }
            if (ok) {
              const uint32_t dst = kp0 + ks * C::KPB + kr * 128;
              if (!has_src) {
#pragma unroll
                for (int u = 0; u < 8; ++u) sts(dst + ((u ^ sw) << 4), make_uint4(0, 0, 0, 0));
              } else if (FP8) {
                const uint32_t src = rbase + roff + (c >> 1) * cs;
                uint4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = lds(src + (((4 * (c & 1) + i) ^ sw) << 4));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  sts(dst + (((2 * i) ^ sw) << 4),
                      make_uint4(e4m3x2_to_f16x2(v[i].x), e4m3x2_to_f16x2(v[i].x >> 16), e4m3x2_to_f16x2(v[i].y),
                                 e4m3x2_to_f16x2(v[i].y >> 16)));
                  sts(dst + (((2 * i + 1) ^ sw) << 4),
                      make_uint4(e4m3x2_to_f16x2(v[i].z), e4m3x2_to_f16x2(v[i].z >> 16), e4m3x2_to_f16x2(v[i].w),
                                 e4m3x2_to_f16x2(v[i].w >> 16)));
                }
              } else {
                const uint32_t src = rbase + roff + c * cs;
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = lds(src + ((u ^ sw) << 4));  // both rows have the same
#pragma unroll                                                                      // swizzle phase: copy units
                for (int u = 0; u < 8; ++u) sts(dst + ((u ^ sw) << 4), v[u]);  // as stored, a bank group each
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBKpFull + ks));
          }
          if (FP8) {  // for the softmax: scale_log2 * K scale, and the V scale
            s_kss[(st & 3) * 128 + kr] = sl * ksc;
            s_vss[(st & 3) * 128 + kr] = vsc_f;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBKssFull + (st & 3)));
          }
        } else {
          // V^T sub-tiles (tt, head hv): this thread writes pieces of row
          // r = kr % TSK (token r of head hv): 32 bytes of output each, PPT
          // of the row's 8 pieces starting at part * PPT.
          constexpr int SUBR = C::SUBR;
          constexpr int PPT = SUBR / 16;
          const int r0 = kr % SUBR, part = kr / SUBR;
          const int swr = r0 & 7;
          for (int tt = 0; tt < NVT; ++tt) {
            for (int hk = 0; hk < H2 * C::NKH; ++hk, ++vti) {
              const int hv = hk / C::NKH;
              const int r = (hk % C::NKH) * SUBR + r0;  // token of head hv
              const bool r_ok = scr ? r < p.T : r < valid;
              const int vsl = vti & 1;
              if (ok && vti >= 2) {
                ok = mbar_wait_sleep(bar(kBVtEmpty + vsl), ((vti >> 1) - 1) & 1, kWaitLimitNs, s_abort);
                if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
              }
              if (ok) {
                const uint32_t srow = rbase + (scr ? (uint32_t)(hv * p.TP * 128 + r * 128)
                                                   : (uint32_t)((r >> p.lbr) * box_bytes + hv * p.BR * 128 +
                                                                (r & (p.BR - 1)) * 128));
                const uint32_t drow = vt0 + vsl * C::SUBB + r0 * 128;
#pragma unroll
                for (int q0 = 0; q0 < PPT; ++q0) {
                  const int q = part * PPT + q0;  // piece: chunk cc = q / 4 of the tile, pair i = q % 4
                  const int cc = q >> 2, i = q & 3;
                  const int c = 2 * tt + cc;      // 64-column chunk of the row
                  const uint32_t dst = drow + cc * (SUBR * 128);
                  uint4 lo, hi;
                  if (!r_ok) {  // past the stage's valid tokens: zero (the product must see no NaN)
                    lo = hi = make_uint4(0, 0, 0, 0);
                  } else if (FP8) {
                    const uint4 v = lds(srow + (c >> 1) * cs + (((4 * (c & 1) + i) ^ swr) << 4));
                    lo = make_uint4(e4m3x2_to_f16x2(v.x), e4m3x2_to_f16x2(v.x >> 16), e4m3x2_to_f16x2(v.y),
                                    e4m3x2_to_f16x2(v.y >> 16));
                    hi = make_uint4(e4m3x2_to_f16x2(v.z), e4m3x2_to_f16x2(v.z >> 16), e4m3x2_to_f16x2(v.w),
                                    e4m3x2_to_f16x2(v.w >> 16));
                  } else {
                    lo = lds(srow + c * cs + (((2 * i) ^ swr) << 4));
                    hi = lds(srow + c * cs + (((2 * i + 1) ^ swr) << 4));
                  }
                  sts(dst + (((2 * i) ^ swr) << 4), lo);
                  sts(dst + (((2 * i + 1) ^ swr) << 4), hi);
                }
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(kBVtFull + vsl));
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar((isK ? kBRawKEmpty : kBRawVEmpty) + slot));
      }
      stage += it.nst;
    }
  } else {
    regs_inc<kRegSoftmax>();
    // ================================================================ softmax
    // warp w < 4: key rows kr = 32 w + lane = token t of head h.
    const int kr = tid;
    const int h = kr / TSK, t = kr % TSK;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const int wh0 = (h * TSK) >> 5, nwh = TSK >> 5;  // this head's softmax warps
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
    float* alpha = reinterpret_cast<float*>(smem + C::OFF_ALPHA);
    float* colL = reinterpret_cast<float*>(smem + C::OFF_COLL);
    float* colM = reinterpret_cast<float*>(smem + C::OFF_COLM);
    const uint32_t pt0 = sbase + C::OFF_PT;
    // The running max moves only past this slack, so p = 2^(s - m) <= 2^slack.
    // fp8: P also carries the token's V scale, p * v_scale in f16; a slack of
    // 4 keeps it finite for V scales up to 4095 (|v| up to 1.8e6).
    constexpr float slack = FP8 ? 4.f : kMaxSlack;
    const float sl = p.scale_log2;
    int stage = 0, oi = 0;

    // Balanced schedule: a sequence with no keys has no work item; CTA
    // b % grid writes its rows (out = 0, lse = -inf).
    if (p.num_splits == 0 && !p.tidar) {
      for (int b = blockIdx.x; b < p.B; b += p.grid) {
        if (s_ctx[b] != 0) continue;
        const size_t rows = (size_t)p.T * p.Hq;
        uint4* o4 = reinterpret_cast<uint4*>(p.out + (size_t)b * rows * D);
        for (size_t i = kr; i < rows * D / 8; i += 128) o4[i] = make_uint4(0, 0, 0, 0);
        if (p.lse)
          for (size_t i = kr; i < rows; i += 128) p.lse[(size_t)b * rows + i] = NEG_INF;
      }
    }

    while (next_item(p, s_ctx, s_start, cur, it)) {
      float m[GT], l[GT];
#pragma unroll
      for (int i = 0; i < GT; ++i) {
        m[i] = NEG_INF;
        l[i] = 0.f;
      }
      // Scratch stage: bit i is set when the query row (column) i of this
      // head sees this thread's scratch token: all T, or the draft-block
      // prefix of a block-masked draft.
      uint64_t vis_bits = 0;
      if (it.scratch) {
#pragma unroll
        for (int i = 0; i < GT; ++i) {
          const int tq = i / p.G;
          if (t < min(p.T, (tq / p.draft_block + 1) * p.draft_block)) vis_bits |= 1ull << i;
        }
      }
      const float* s_kss = reinterpret_cast<const float*>(smem + C::OFF_KSS);
      const float* s_vss = reinterpret_cast<const float*>(smem + C::OFF_VSS);
      const int ob = oi & 1;

      for (int j = 0; j < it.nst; ++j) {
        const int st = stage + j, sb = st & 1;
        float s[GT];
        if (ok) {
          ok = mbar_wait_sleep(bar(kBSFull + sb), (st >> 1) & 1, kWaitLimitNs, s_abort);
          if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
        }
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok)) {
          tmem_ld<GT>(tm + lane_base + (uint32_t)(sb * N + h * GT), s);
        } else {
#pragma unroll
          for (int i = 0; i < GT; ++i) s[i] = 0.f;
        }
        // fp8: this row's scale_log2 * K scale and V scale (slot st % 4: the
        // K converters run at most two stages ahead of this read)
        float kss = sl, vsr = 1.f;
        if (FP8) {
          if (ok) {
            ok = mbar_wait_sleep(bar(kBKssFull + (st & 3)), (st >> 2) & 1, kWaitLimitNs, s_abort);
            if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
          }
          kss = s_kss[(st & 3) * 128 + kr];
          vsr = s_vss[(st & 3) * 128 + kr];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBSEmpty + sb));
        // scale (and the K scale of this row's token), mask
        const bool scr = it.scratch && j == it.nst - 1;
        const int valid = scr ? p.T : min(TSK, it.tok_end - (it.tok0 + j * TSK));
        if (scr) {
#pragma unroll
          for (int i = 0; i < GT; ++i) s[i] = (vis_bits >> i) & 1 ? s[i] * kss : NEG_INF;
        } else {
          const bool tv = t < valid;
#pragma unroll
          for (int i = 0; i < GT; ++i) s[i] = tv ? s[i] * kss : NEG_INF;
        }
        // stage max of every column over the head's tokens: the warp's by
        // one reduction per column, then across the head's warps through
        // shared memory (mn holds the maxima, then the new running max)
        float mn[GT];
#pragma unroll
        for (int i = 0; i < GT; ++i) mn[i] = redux_max(s[i]);
        if (nwh > 1) {
          if (lane == 0) {
#pragma unroll
            for (int i = 0; i < GT; i += 4)
              *reinterpret_cast<float4*>(red + warp * 64 + i) = make_float4(mn[i], mn[i + 1], mn[i + 2], mn[i + 3]);
          }
          named_barrier_sync(1, 128);
#pragma unroll
          for (int w2 = 0; w2 < nwh; ++w2) {
            if (wh0 + w2 == warp) continue;
#pragma unroll
            for (int i = 0; i < GT; i += 4) {
              const float4 x = *reinterpret_cast<const float4*>(red + (wh0 + w2) * 64 + i);
              mn[i] = fmaxf(mn[i], x.x);
              mn[i + 1] = fmaxf(mn[i + 1], x.y);
              mn[i + 2] = fmaxf(mn[i + 2], x.z);
              mn[i + 3] = fmaxf(mn[i + 3], x.w);
            }
          }
        }
        bool need_o = false;
#pragma unroll
        for (int i = 0; i < GT; ++i) {
          mn[i] = mn[i] > m[i] + slack ? mn[i] : m[i];
          need_o |= (m[i] != NEG_INF) && (mn[i] != m[i]);
        }
        if (named_barrier_or(2, 128, need_o)) {
          // A running max moved: rescale l and the O^T columns (all heads:
          // O^T rows are head-dim lanes, spread over the four quadrants).
#pragma unroll
          for (int i = 0; i < GT; ++i) {
            const float a = mn[i] == m[i] ? 1.f : (m[i] == NEG_INF ? 0.f : ex2(m[i] - mn[i]));
            l[i] *= a;
            if (warp == wh0 && (i & 31) == lane) alpha[h * GT + i] = a;
          }
          named_barrier_sync(1, 128);
          if (j > 0) {
            if (ok) {
              ok = mbar_wait_sleep(bar(kBPEmpty + (st - 1) % NPT), ((st - 1) / NPT) & 1, kWaitLimitNs, s_abort);
              if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
            }
            tc_fence_after();
            if (__all_sync(0xffffffffu, ok)) {
#pragma unroll
              for (int tt = 0; tt < NVT; ++tt) {
#pragma unroll
                for (int c0 = 0; c0 < N; c0 += 16) {
                  float o[16];
                  const uint32_t oa = tm + lane_base + (uint32_t)(C::TM_O + (ob * NVT + tt) * N + c0);
                  tmem_ld16(oa, o);
#pragma unroll
                  for (int c = 0; c < 16; ++c) o[c] *= alpha[c0 + c];
                  tmem_st16(oa, o);
                }
              }
              tmem_wait_st();
            }
            tc_fence_before();
          }
          named_barrier_sync(1, 128);
        }
#pragma unroll
        for (int i = 0; i < GT; ++i) m[i] = mn[i];
        // p = 2^(s - m) in the MMA's 16-bit type
        uint32_t pk[GT / 2];
#pragma unroll
        for (int i = 0; i < GT; i += 2) {
          const float mu0 = m[i] == NEG_INF ? 0.f : m[i];
          const float mu1 = m[i + 1] == NEG_INF ? 0.f : m[i + 1];
          const float p0 = ex2(s[i] - mu0), p1 = ex2(s[i + 1] - mu1);
          l[i] += p0;
          l[i + 1] += p1;
          pk[i / 2] = FP8 ? pack16<true>(p0 * vsr, p1 * vsr) : pack16<!C::BF16>(p0, p1);
        }
        // P^T row of this token: wait until the product that last read the
        // buffer is done
        const int pb = st % NPT;
        if (ok && st >= NPT) {
          ok = mbar_wait_sleep(bar(kBPEmpty + pb), ((st - NPT) / NPT) & 1, kWaitLimitNs, s_abort);
          if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
        }
        {
          const uint32_t rowa = pt0 + pb * C::PB + h * C::PH + (t >> 3) * (8 * C::PSW) + (t & 7) * C::PSW;
          const int swp = (t & 7) >> C::PSHIFT;
#pragma unroll
          for (int u = 0; u < C::PSW / 16; ++u)
            sts(rowa + ((u ^ swp) << 4), make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBPFull + pb));
      }
      stage += it.nst;

      // ---- epilogue: column sums of l over the head's tokens, then O^T / L
      warp_columns_reduce<GT, false>(l, lane);
      {
        const int c0 = reduced_col0<GT>(lane);
        if (GT != 16 || (lane & 1) == 0) {
#pragma unroll
          for (int r = 0; r < (GT > 32 ? GT / 32 : 1); ++r) red[warp * 64 + c0 + r] = l[r];
        }
        if (warp == wh0) {
#pragma unroll
          for (int i = 0; i < GT; ++i)
            if ((i & 31) == lane) colM[h * GT + i] = m[i];
        }
      }
      named_barrier_sync(1, 128);
      if (kr < N) {
        const int hh = kr / GT, i = kr % GT;
        const int w0 = (hh * TSK) >> 5;
        float L = 0.f;
        for (int w2 = 0; w2 < nwh; ++w2) L += red[(w0 + w2) * 64 + i];
        colL[kr] = L;
      }
      named_barrier_sync(1, 128);
      const bool bad = __any_sync(0xffffffffu, !ok || *s_abort);
      const float NaN = __int_as_float(0x7fffffff);
      if (it.nst > 0) {
        if (ok) {
          ok = mbar_wait_sleep(bar(kBOFull + ob), (oi >> 1) & 1, kWaitLimitNs, s_abort);
          if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
        }
        tc_fence_after();
      }
      const bool bad2 = bad || __any_sync(0xffffffffu, !ok);
#pragma unroll
      for (int tt = 0; tt < NVT; ++tt) {
        const int d = tt * 128 + 32 * warp + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < N; c0 += 16) {
         float o[16];
         if (it.nst > 0 && !bad2) {
           tmem_ld16(tm + lane_base + (uint32_t)(C::TM_O + (ob * NVT + tt) * N + c0), o);
         } else {
#pragma unroll
           for (int c = 0; c < 16; ++c) o[c] = 0.f;
         }
#pragma unroll
         for (int cc = 0; cc < 16; ++cc) {
          const int c = c0 + cc;
          const float L = colL[c];
          float v = L > 0.f ? o[cc] / L : 0.f;
          if (bad2) v = NaN;
          // column c = query row rho -> (head hl, draft token tq, group member jg)
          const int hl = c / GT, rem = c % GT;
          const int tq = rem / p.G;
          const int head = (it.hg * H2 + hl) * p.G + (rem - tq * p.G);
          const size_t row = ((size_t)it.b * p.T + tq) * p.Hq + head;
          if (it.part < 0) {
            __nv_bfloat16* o16 = p.out + row * D + d;
            if (C::BF16 || FP8) {
              *o16 = __float2bfloat16_rn(v);
            } else {
              *reinterpret_cast<__half*>(o16) = __float2half_rn(v);
            }
          } else {
            const size_t prow = p.num_splits > 0 ? row * p.num_splits + it.part : (size_t)it.part * p.M + c;
            p.part_o[prow * D + d] = v;
          }
         }
        }
      }
      if (it.nst > 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBOEmpty + ob));
        ++oi;
      }
      if (kr < N) {
        const int c = kr;
        const float L = colL[c], M = colM[c];
        float lsev = L > 0.f ? (M + lg2(L)) * kLn2 : NEG_INF;
        if (bad2 && it.nst > 0) lsev = NaN;
        const int hl = c / GT, rem = c % GT;
        const int tq = rem / p.G;
        const int head = (it.hg * H2 + hl) * p.G + (rem - tq * p.G);
        const size_t row = ((size_t)it.b * p.T + tq) * p.Hq + head;
        if (it.part < 0) {
          if (p.lse) p.lse[row] = lsev;
        } else {
          const size_t prow = p.num_splits > 0 ? row * p.num_splits + it.part : (size_t)it.part * p.M + c;
          p.part_lse[prow] = lsev;
        }
      }
      named_barrier_sync(1, 128);  // colL / colM / red reused by the next item
    }
  }
  launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == kUMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, C::TM_COLS);
  }
}

}  // namespace pa
