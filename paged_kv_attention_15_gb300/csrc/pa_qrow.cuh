// Query-row-major tcgen05 decode kernel for 16-bit KV caches (bf16, f16)
// and work units of M = 64 query rows (two kv heads of 32 query rows or one
// kv head of 64: grouped heads times draft tokens, the draft-block
// workloads) or M = 128 (four kv heads of 32).
//
// Sources: ROCm blog "Implementing a High-Performance Custom Diffusion
// Attention Kernel with FlyDSL" (introduction items 1-3: head packing into
// the matrix-core M dimension, online softmax, prefetched loads) and the MSLK
// pull request "[ROCm] Add FlyDSL paged-attention decode backend (dense +
// fp8) with benchmark" (Kernels: head-packed decode over the block table,
// split-K partials combined by log-sum-exp). Same operation, schedule and
// outputs as the warp-level split kernel (pa_kernels.cuh); the arithmetic is
// laid out for the fifth-generation tensor cores:
//
//  - a stage tile is [chunk][key row][128 B] with the stage's 64 key rows
//    (page box, head, row) contiguous in every chunk, 128-byte swizzled: for
//    M = 64 the producer copies each page once per 128-byte column chunk;
//    for M = 128 a stage is one 16-token page box of the four heads, which
//    has that layout already and is copied whole;
//  - S = Q K^T per stage with M = the unit's query rows (tcgen05.mma,
//    kind::f16, fp32 accumulator in tensor memory), one MMA per 16-column
//    k-step over all the stage's key rows (N = up to 64): the B descriptor
//    points straight into the TMA-landed K tile, so K is never copied;
//  - softmax in warps 0-3: with M = 64 the accumulator row i sits in tensor
//    memory lane 32 (i / 16) + i % 16, so lane l < 16 of warp w owns query
//    row 16 w + l (M = 128: row i in lane i, lane l of warp w owns row
//    32 w + l) and reads only its own kv head's score columns; the row
//    max and sum are thread-local (no cross-thread reduction), the running
//    max moves lazily (kMaxSlack), and the thread writes its row of P (16-bit,
//    zeros in the other head's columns) into a 128-byte-swizzled K-major tile;
//  - O += P V with N = D, one MMA per 16 key rows: V is the B operand
//    in its landed layout (MN-major: dims contiguous, LBO = the chunk stride,
//    SBO = 8 key rows), O stays in tensor memory for the whole work item and
//    is read once by the epilogue (O / l, and the log-sum-exp);
//  - a producer warp fills the stage ring like the warp-level kernel
//    (produce_ring), one MMA warp issues both products:
//    S of stage j, then P V of stage j - 1, so the softmax of stage j
//    overlaps P V of j - 1. (A tcgen05.mma has a fixed cost of tens of
//    cycles however small its N: a stage takes D / 16 + 4 of them.)
// Key rows of the last page past the context are zeroed in shared memory
// before P V reads them (P is 0 there, and 0 * NaN must not reach O). Every
// wait is bounded; an item cut short is written as NaN.
#pragma once

#include "pa_kernels.cuh"
#include "pa_tc.cuh"

namespace pa {

constexpr int kQThreads = 192;  // softmax warps 0-3, producer warp 4, MMA warp 5
constexpr int kQProducerWarp = 4;
constexpr int kQMmaWarp = 5;

// M = 64: two kv heads of 32 query rows or one of 64, pages copied per
// 128-byte chunk, two Q slots. M = 128: four kv heads of 32 rows, whose
// 16-token page box already holds the stage's 64 key rows contiguously in
// every chunk (one copy per page, a 16 KB box), one Q slot (the ring keeps
// four stages).
template <int D, int M_>
struct QCfg {
  static constexpr int M = M_;        // query rows of a unit: the MMA M
  static constexpr bool CB = M == 64; // one copy per page and chunk (else per page)
  static constexpr int NQ = M == 128 ? 1 : 2;  // Q slots
  static constexpr int KR = 64;       // key rows (tokens x heads) of a stage
  static constexpr int NCH = D / 64;  // 128-byte column chunks of a 16-bit row
  static constexpr int TILE = KR * D * 2;  // [chunk][key row][128 B]
  static constexpr int CSTR = KR * 128;     // chunk stride of a tile
  static constexpr int STAGE = 2 * TILE;
  static constexpr int QCHUNK = M * 128;
  static constexpr int QSLOT = NCH * QCHUNK;
  static constexpr int PBUF = M * KR * 2;  // P of a stage: one 128-byte row (64 keys) per query row
  static constexpr int NPB = 2;
  static constexpr int BARS = 256;
  static constexpr int FIXED = NQ * QSLOT + NPB * PBUF + BARS + 64;
  static constexpr int NS = clamp_int((kSmemBudget - FIXED) / STAGE, 2, 8);
  static constexpr int OFF_Q = NS * STAGE;
  static constexpr int OFF_P = OFF_Q + NQ * QSLOT;
  static constexpr int OFF_BAR = OFF_P + NPB * PBUF;
  static constexpr int OFF_MISC = OFF_BAR + BARS;  // tensor-memory base, abort flag
  static constexpr int OFF_TABLE = OFF_MISC + 64;
  static constexpr int SMEM_FIXED = OFF_TABLE + 1024;  // + 1024 to align the dynamic base
  static constexpr int TM_S = 0;                       // [2][KR] score columns
  static constexpr int TM_O = 2 * KR;                  // [D] output columns
  static constexpr int TM_COLS = 2 * KR + D <= 256 ? 256 : 512;
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(M == 64 || M == 128, "query rows per unit");
  static_assert(2 * NS + 16 <= BARS / 8, "barriers");
};

// Barriers after the ring's full[NS] and empty[NS]: Q slots (full, empty),
// score buffers (full, empty), P buffers (full, empty), O (full, empty),
// the completion of each P V product, and the MMA warp's final drain.
enum : int {
  kQbQFull = 0,
  kQbQEmpty = 2,
  kQbSFull = 4,
  kQbSEmpty = 6,
  kQbPFull = 8,
  kQbPEmpty = 10,
  kQbOFull = 12,
  kQbOEmpty = 13,
  kQbPvDone = 14,
  kQbDone = 15,
};

// Page boxes of a stage (the layout the producer wrote): `nbox` boxes of
// `brows` rows per head (brows = 2^lb); the draft-token scratch is one box
// of TP rows.
struct QStage {
  int nbox, brows, lb, valid;  // valid: paged tokens of the stage (per head), or T for the scratch
  bool scr;
};

__device__ __forceinline__ QStage q_stage(const SplitParams& p, const Item& it, int j) {
  QStage g;
  g.scr = it.scratch && j == it.nst - 1;
  if (g.scr) {
    g.nbox = 1;
    g.brows = p.TP;
    g.valid = p.T;
  } else {
    g.valid = min(p.TS, it.tok_end - (it.tok0 + j * p.TS));
    g.brows = p.BR;
    g.nbox = p.P < p.TS ? (g.valid + p.P - 1) >> p.lbr : 1;
  }
  g.lb = 31 - __clz(g.brows);
  return g;
}

template <int D, int KV, int H2, int M>
__global__ void __launch_bounds__(kQThreads, 1) pa_qrow_kernel(const __grid_constant__ SplitParams p) {
  using C = QCfg<D, M>;
  constexpr int NQ = C::NQ;
  constexpr int LH2 = H2 == 4 ? 2 : (H2 == 2 ? 1 : 0);  // log2 of H2
  constexpr bool F16 = KV == kKvF16;
  constexpr int NS = C::NS;
  constexpr int KR = C::KR;
  constexpr int OWN = KR / H2;  // score columns of one kv head per stage
  constexpr int NOG = OWN / 16; // ... in groups of 16
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t bar_full = sbase + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * NS;
  const uint32_t bq = bar_full + 16 * NS;
  auto bar = [&](int i) { return bq + 8u * (uint32_t)i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  int* s_ctx = reinterpret_cast<int*>(smem + C::OFF_TABLE);
  int* s_start = s_ctx + (p.num_splits == 0 ? p.B : 0);
  const float NEG_INF = -__int_as_float(0x7f800000);

  if (tid == 32 * kQProducerWarp) prefetch_maps(p);  // the producer's lane 0
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kQbQFull + s), 1);
      mbar_init(bar(kQbQEmpty + s), 1);
      mbar_init(bar(kQbSFull + s), 1);
      mbar_init(bar(kQbSEmpty + s), 4);
      mbar_init(bar(kQbPFull + s), 4);
      mbar_init(bar(kQbPEmpty + s), 1);
    }
    mbar_init(bar(kQbOFull), 1);
    mbar_init(bar(kQbOEmpty), 4);
    mbar_init(bar(kQbPvDone), 1);
    mbar_init(bar(kQbDone), 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  {  // query rows past M read as zero: clear the Q slots once
    uint4* q4 = reinterpret_cast<uint4*>(smem + C::OFF_Q);
    for (int i = tid; i < NQ * C::QSLOT / 16; i += kQThreads) q4[i] = make_uint4(0, 0, 0, 0);
  }
  if (warp == kQMmaWarp) tmem_alloc(sbase + C::OFF_MISC, C::TM_COLS);
  if (p.num_splits == 0) {
    for (int i = tid; i < p.B; i += kQThreads) s_ctx[i] = clamp_ctx(p, __ldg(p.context_lens + i));
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
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *s_tmem;

  if (warp == kQProducerWarp) {
    // ================================================================ producer
    const RingGeom g{sbase, (uint32_t)C::OFF_Q, (uint32_t)C::QSLOT, (uint32_t)C::QCHUNK, (uint32_t)C::STAGE,
                     (uint32_t)C::TILE, NS, C::NCH, C::NCH, (uint32_t)(H2 * D * 2),
                     C::CB ? (uint32_t)C::CSTR : 0u, NQ};
    produce_ring(p, s_ctx, s_start, g, bar_full, bar_empty, bar(kQbQFull), bar(kQbQEmpty), s_abort, lane);
  } else if (warp == kQMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t id_pv = idesc_f16(C::M, D, !F16, false, true);
      Cursor cur;
      cursor_init(p, s_start, cur);
      Item it;
      int stage = 0, qn = 0, items = 0;
      bool ok = true;
      while (ok && next_item(p, s_ctx, s_start, cur, it)) {
        if (it.nst == 0) continue;
        const int qs = qn % NQ;
        ok = mbar_wait(bar(kQbQFull + qs), (qn / NQ) & 1, kWaitLimitNs, s_abort);
        const uint32_t qbase = sbase + C::OFF_Q + qs * C::QSLOT;
        for (int j = 0; ok && j <= it.nst; ++j) {
          if (j < it.nst) {
            // ---- S(j) = Q K^T into score buffer st & 1
            const int st = stage + j, slot = st % NS, sb = st & 1;
            ok = mbar_wait(bar_full + 8 * slot, (st / NS) & 1, kWaitLimitNs, s_abort);
            if (ok && st >= 2) ok = mbar_wait(bar(kQbSEmpty + sb), ((st >> 1) - 1) & 1, kWaitLimitNs, s_abort);
            if (!ok) break;
            tc_fence_after();
            const QStage g = q_stage(p, it, j);
            const int nkeys = g.nbox * H2 * g.brows;  // key rows of the stage (a multiple of 16)
            const uint32_t cs = C::CB ? (uint32_t)C::CSTR : (uint32_t)nkeys * 128u;  // chunk stride
            const uint32_t id_s = idesc_f16(C::M, nkeys, !F16, false, false);
            const uint32_t kb = sbase + slot * C::STAGE;
            const uint32_t d_s = tm + (uint32_t)(C::TM_S + sb * KR);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint64_t a = smem_desc(qbase + (ks >> 2) * C::QCHUNK + (ks & 3) * 32, 16, 1024, kSwz128);
              const uint64_t b = smem_desc(kb + (ks >> 2) * cs + (ks & 3) * 32, 16, 1024, kSwz128);
              umma_f16(d_s, a, b, id_s, ks > 0 ? 1u : 0u);
            }
            umma_commit(bar(kQbSFull + sb));
            if (j == it.nst - 1) umma_commit(bar(kQbQEmpty + qs));
          }
          if (j >= 1) {
            // ---- O += P(j-1) V(j-1)
            const int jj = j - 1, st = stage + jj, slot = st % NS, pb = st & 1;
            ok = mbar_wait(bar(kQbPFull + pb), (st >> 1) & 1, kWaitLimitNs, s_abort);
            if (ok && jj == 0 && items > 0) ok = mbar_wait(bar(kQbOEmpty), (items - 1) & 1, kWaitLimitNs, s_abort);
            if (!ok) break;
            tc_fence_after();
            const QStage g = q_stage(p, it, jj);
            const int nkeys = g.nbox * H2 * g.brows;
            const uint32_t cs = C::CB ? (uint32_t)C::CSTR : (uint32_t)nkeys * 128u;
            const uint32_t vb = sbase + slot * C::STAGE + C::TILE;
            const uint32_t pbuf = sbase + C::OFF_P + pb * C::PBUF;
            for (int key = 0; key < nkeys; key += 16) {  // P columns of the k-step
              const uint64_t a = smem_desc(pbuf + (key >> 4) * 32, 16, 1024, kSwz128);
              const uint64_t b = smem_desc(vb + key * 128, cs, 1024, kSwz128);
              umma_f16(tm + C::TM_O, a, b, id_pv, (jj > 0 || key > 0) ? 1u : 0u);
            }
            umma_commit(bar_empty + 8 * slot);
            umma_commit(bar(kQbPEmpty + pb));
            umma_commit(bar(kQbPvDone));
            if (jj == it.nst - 1) umma_commit(bar(kQbOFull));
          }
        }
        stage += it.nst;
        ++qn;
        ++items;
      }
      if (!ok) raise_abort(s_abort, p.err_flags);
      // Every product issued has completed before tensor memory is freed.
      umma_commit(bar(kQbDone));
      const int zero = 0;
      mbar_wait(bar(kQbDone), 0, kWaitLimitNs, &zero);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax + epilogue
    const int GT = p.GT;
    // M = 64: row i in lane 32 (i / 16) + i % 16, so lane l < 16 of warp w
    // owns row 16 w + l (lanes >= 16 mirror 0-15); M = 128: lane l of warp w
    // owns row 32 w + l.
    const bool act = M == 128 || lane < 16;
    const int rho = M == 128 ? 32 * warp + lane : 16 * warp + (lane & 15);
    const int hl = rho / GT;  // its kv head in the unit (warp-uniform: GT >= 16 / 32)
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float sl = p.scale_log2;
    // Draft tokens the row's draft token sees in the scratch: all T, or the
    // draft-block prefix of a block-masked draft.
    const int tq = (rho % GT) / p.G;
    const int vis = min(p.T, (tq / p.draft_block + 1) * p.draft_block);

    // Balanced schedule: a sequence with no keys has no work item; CTA
    // b % grid writes its rows (out = 0, lse = -inf).
    if (p.num_splits == 0 && !p.tidar) {
      for (int b = blockIdx.x; b < p.B; b += p.grid) {
        if (s_ctx[b] != 0) continue;
        const size_t rows = (size_t)p.T * p.Hq;
        uint4* o4 = reinterpret_cast<uint4*>(p.out + (size_t)b * rows * D);
        for (size_t i = tid; i < rows * D / 8; i += 128) o4[i] = make_uint4(0, 0, 0, 0);
        if (p.lse)
          for (size_t i = tid; i < rows; i += 128) p.lse[(size_t)b * rows + i] = NEG_INF;
      }
    }

    Cursor cur;
    cursor_init(p, s_start, cur);
    Item it;
    int stage = 0, items = 0;
    bool ok = true;
    while (next_item(p, s_ctx, s_start, cur, it)) {
      float m = NEG_INF, l = 0.f;
      for (int j = 0; j < it.nst; ++j) {
        const int st = stage + j, sb = st & 1, pb = st & 1, slot = st % NS;
        if (ok) {
          ok = mbar_wait(bar(kQbSFull + sb), (st >> 1) & 1, kWaitLimitNs, s_abort);
          if (!ok) raise_abort(s_abort, p.err_flags);
        }
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        const QStage g = q_stage(p, it, j);
        const int nrows = H2 * g.brows;     // key rows of a page box (all heads)
        const int lbn = g.lb + LH2;         // log2 of nrows
        const int nown = g.nbox * g.brows;  // own score columns written this stage
        // ---- this head's score columns, 16 at a time: own slot o = token
        // (paged: box o / brows, row o % brows; scratch: draft token o)
        float s[OWN];
#pragma unroll
        for (int q = 0; q < NOG; ++q) {
          const int o0 = 16 * q;
          if (ok && o0 < nown) {
            const int i = o0 >> g.lb, r0 = o0 & (g.brows - 1);
            tmem_ld16(tm + lane_base + (uint32_t)(C::TM_S + sb * KR + i * nrows + hl * g.brows + r0), s + o0);
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) s[o0 + c] = NEG_INF;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kQbSEmpty + sb));

        // ---- scale, mask, online softmax in base 2 (one row per thread)
        const int lim = g.scr ? min(vis, g.brows) : g.valid;
        float mx = NEG_INF;
#pragma unroll
        for (int o = 0; o < OWN; ++o) {
          s[o] = o < lim ? s[o] * sl : NEG_INF;
          mx = fmaxf(mx, s[o]);
        }
        const float mn = mx > m + kMaxSlack ? mx : m;
        const float mu = mn == NEG_INF ? 0.f : mn;
        const float al = mn == m ? 1.f : ex2(m - mu);
        m = mn;
        float ls = 0.f;
        uint32_t pk[OWN / 2];
#pragma unroll
        for (int o = 0; o < OWN; o += 2) {
          const float p0 = ex2(s[o] - mu), p1 = ex2(s[o + 1] - mu);
          ls += p0 + p1;
          pk[o / 2] = pack16<F16>(p0, p1);
        }
        l = l * al + ls;

        // ---- the running max moved past the slack (rare): rescale O once
        // the previous stage's product has landed
        if (__any_sync(0xffffffffu, act && j > 0 && al != 1.f) && ok) {
          ok = mbar_wait(bar(kQbPvDone), (st - 1) & 1, kWaitLimitNs, s_abort);
          if (!ok) raise_abort(s_abort, p.err_flags);
          if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const float f = act ? al : 1.f;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 16) {
              float o[16];
              tmem_ld16(tm + lane_base + (uint32_t)(C::TM_O + c0), o);
#pragma unroll
              for (int c = 0; c < 16; ++c) o[c] *= f;
              tmem_st16(tm + lane_base + (uint32_t)(C::TM_O + c0), o);
            }
            tmem_wait_st();
          }
          ok = __all_sync(0xffffffffu, ok);
        }

        // ---- P row: 64 keys in the stage's key order (box, head, row);
        // this head's keys carry p, the other head's are zero
        if (ok && st >= 2) {
          ok = mbar_wait(bar(kQbPEmpty + pb), ((st >> 1) - 1) & 1, kWaitLimitNs, s_abort);
          if (!ok) raise_abort(s_abort, p.err_flags);
        }
        ok = __all_sync(0xffffffffu, ok);
        if (act && ok) {
          const uint32_t prow = sbase + C::OFF_P + pb * C::PBUF + (uint32_t)rho * 128u;
#pragma unroll
          for (int kg = 0; kg < KR / 16; ++kg) {  // key group: keys 16 kg .. 16 kg + 15
            uint32_t v[8];
            if (H2 == 1) {
#pragma unroll
              for (int u = 0; u < 8; ++u) v[u] = pk[kg * 8 + u];
            } else {
              // head of the group and own group index: boxes of nrows keys
              // (paged: brows >= 16), or the scratch's 8-key heads (two per
              // group)
              if (g.scr && g.brows == 8) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  v[u] = (kg == (hl >> 1) && (u >> 2) == (hl & 1)) ? pk[u & 3] : 0u;
              } else {
                const int key = 16 * kg;
                const int i = key >> lbn, w = key & (nrows - 1);
                const int h = w >> g.lb;
                const int og = ((i << g.lb) + (w & (g.brows - 1))) >> 4;  // own 16-slot group
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  uint32_t x = 0u;
#pragma unroll
                  for (int q = 0; q < NOG; ++q) x = og == q ? pk[q * 8 + u] : x;
                  v[u] = (h == hl && i < g.nbox) ? x : 0u;
                }
              }
            }
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
              const int unit = 2 * kg + u2;
              st_shared_v4(prow + (uint32_t)(((unit ^ (rho & 7)) << 4)),
                           make_uint4(v[4 * u2], v[4 * u2 + 1], v[4 * u2 + 2], v[4 * u2 + 3]));
            }
          }
        }
        // ---- last page of the item: key rows past the context are zeroed
        // in the V tile (all 128 threads of the four warps share the rows)
        if (ok && !g.scr && g.valid < g.nbox * g.brows) {
          const uint32_t vb = sbase + slot * C::STAGE + C::TILE;
          const int last = g.nbox - 1;                        // the partial box
          const int r_lo = g.valid - last * g.brows;          // its first row past the context
          const int nr = g.brows - r_lo;
          const int nz = nr * H2 * C::NCH * 8;                // 16-byte units to clear
          for (int u = tid; u < nz; u += 128) {
            const int unit = u & 7, rest = u >> 3;
            const int r = r_lo + rest % nr;
            const int hc = rest / nr;  // head + H2 * chunk
            const int h = hc % H2, c = hc / H2;
            const uint32_t cs = C::CB ? (uint32_t)C::CSTR : (uint32_t)(g.nbox * nrows) * 128u;
            const uint32_t row_addr = vb + (uint32_t)c * cs + (uint32_t)(last * nrows + h * g.brows + r) * 128u;
            st_shared_v4(row_addr + (uint32_t)(unit << 4), make_uint4(0, 0, 0, 0));
          }
        }
        fence_proxy_async_smem();  // P (and zeroed rows) -> the tensor core's reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kQbPFull + pb));
      }
      stage += it.nst;

      // ---- epilogue: O / l and the log-sum-exp of this row
      if (it.nst > 0) {
        if (ok) {
          ok = mbar_wait(bar(kQbOFull), items & 1, kWaitLimitNs, s_abort);
          if (!ok) raise_abort(s_abort, p.err_flags);
        }
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
      }
      const bool bad = __any_sync(0xffffffffu, !ok || *s_abort);
      const float NaN = __int_as_float(0x7fffffff);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float lsev = l > 0.f ? (m + lg2(l)) * kLn2 : NEG_INF;
      if (bad) lsev = NaN;
      // row rho = hl * GT + t * G + j  ->  query head (hg * H2 + hl) * G + j
      const int rem = rho - hl * GT;
      const int t = rem / p.G;
      const int h = (it.hg * H2 + hl) * p.G + (rem - t * p.G);
      const size_t row = ((size_t)it.b * p.T + t) * p.Hq + h;
      const bool write = act && rho < p.M;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float o[16];
        if (it.nst > 0 && !bad) {
          tmem_ld16(tm + lane_base + (uint32_t)(C::TM_O + c0), o);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) o[c] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) o[c] = bad ? NaN : o[c] * inv;
        if (!write) continue;
        if (it.part < 0) {
          uint4* o16 = reinterpret_cast<uint4*>(p.out + row * D + c0);
          uint32_t w[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) w[c] = pack16<F16>(o[2 * c], o[2 * c + 1]);
          o16[0] = make_uint4(w[0], w[1], w[2], w[3]);
          o16[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          const size_t prow = p.num_splits > 0 ? row * p.num_splits + it.part : (size_t)it.part * p.M + rho;
          float4* o32 = reinterpret_cast<float4*>(p.part_o + prow * D + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c) o32[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        }
      }
      if (write) {
        if (it.part < 0) {
          if (p.lse) p.lse[row] = lsev;
        } else {
          const size_t prow = p.num_splits > 0 ? row * p.num_splits + it.part : (size_t)it.part * p.M + rho;
          p.part_lse[prow] = lsev;
        }
      }
      if (it.nst > 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kQbOEmpty));
        ++items;
      }
    }
  }
  launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == kQMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, C::TM_COLS);
  }
}

}  // namespace pa
