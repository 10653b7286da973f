// Paged-KV decode attention kernels for sm_103a.
//
// The split kernel computes softmax attention of the query rows of H2
// consecutive kv heads (head packing: the GQA group times the draft tokens,
// times H2 kv heads, form the MMA M dimension) over a contiguous range of
// one sequence's paged keys, FlashAttention style: online max and sum in
// base 2, rescaled accumulator, and a log-sum-exp per row. A row only sees
// the keys of its own kv head (block-diagonal mask). The reduce kernels
// merge split-K partials by their log-sum-exp.
// Sources: ROCm blog "Implementing a High-Performance Custom Diffusion
// Attention Kernel with FlyDSL" (introduction items 1-3; "Match MFMA Operands
// to the Desired Fragment Layout": the score fragment feeds the P x V
// product without a trip through shared memory; "Prefetch Data"; "Address
// LDS Bank Conflicts") and the MSLK pull request "[ROCm] Add FlyDSL
// paged-attention decode backend (dense + fp8) with benchmark" (Kernels:
// head-packed matrix-core decode with double-buffered loads, native fp8
// e4m3fn KV with symmetric per-token scale, split-K partial combine).
//
// GB300 design. One CTA per SM (persistent) or per (sequence, head group,
// split). The last warp produces: it walks the block table and issues one
// TMA box per page and stage (every column chunk of the page's rows of H2
// kv heads) into a ring of NS shared-memory stages of 64 key rows (64/H2
// tokens x H2 heads), each guarded by a pair of mbarriers (full: bytes
// landed; empty: consumers done). H2 is chosen so a 16-row page still makes
// a large box: small boxes cannot keep enough bytes in flight per SM. The
// other warps consume the ring in order: warp w takes row tile w % MT and,
// inside it, one kv head and one token slice of every stage (or of every
// other stage), keeping its own online-softmax state. fp8 consumers also
// copy their tokens' scales into a small per-warp ring themselves, a few
// stages ahead (4-byte asynchronous copies).
// QK^T and PV run as mma.sync m16n8k16 with fp32 accumulators; the score
// fragment becomes the P operand in registers; K is read with ldmatrix and
// V with ldmatrix.trans from 128-byte-swizzled tiles (conflict-free). At
// the end of a work item the warps of a row tile merge through shared
// memory. Every wait is bounded in time, so a protocol error cannot hang
// the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "pa_ptx.cuh"

namespace pa {

constexpr int kConsumerWarps = 4;  // consumer warps of most instances (one per SM sub-partition)
// Capacity in key rows (tokens x heads) of a pipeline stage: 64, or 128
// for the 128-byte rows of 16-bit D = 64 and 32 for the 512-byte rows of
// 16-bit D = 256, so that a stage's K tile is 16 KB: the per-stage waits and
// arrivals spread over as many bytes, and D = 256 keeps five stages in the
// ring instead of two of 64 KB.
// The host picks the rows a launch actually uses per stage (p.TS * H2).
constexpr int stage_rows(int row_bytes, bool fp8) {
  return fp8 ? 64 : (row_bytes <= 128 ? 128 : (row_bytes >= 512 ? 32 : 64));
}
constexpr int kSmemBudget = 220 * 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kErrWaitTimeout = 1;
constexpr float kLn2 = 0.69314718055994530942f;
// 16-bit pages: the running row max of the online softmax moves only when a
// score passes it by more than this (log2 units). Probabilities 2^(s - m)
// stay below 2^8, well inside f16 and bf16, and the accumulator is rescaled
// a few times per row instead of at every new maximum; l and the
// accumulator share m, so the result is the same up to rounding. (fp8 keeps
// the exact max: its P operand also carries the V scale, in f16.)
constexpr float kMaxSlack = 8.f;
// fp8: a consumer warp copies the scales of a stage this many handled
// stages before it uses them (and keeps one more slot for the stage in use).
constexpr int kScaleAhead = 2;
constexpr int kScaleRing = kScaleAhead + 1;
// Eight consumer warps with long slices (or fp8): 12 warps launch at 168
// registers (the limit of three warps on one SM sub-partition); the
// producer's warpgroup (the producer and three idle warps) drops to 40 and
// the two consumer warpgroups rise to 232, room for a 32-token score slice
// next to the output rows with two consumer warps per sub-partition:
// 2 x 128 x 232 + 128 x 40 = 384 x 168.
constexpr int kSplitLaunchRegs = 168, kSplitConsumerRegs = 232, kSplitProducerRegs = 40;
static_assert(2 * 128 * kSplitConsumerRegs + 128 * kSplitProducerRegs <= 384 * kSplitLaunchRegs,
              "register split exceeds the launch pool");

constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }
constexpr int clamp_int(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

struct SplitParams {
  CUtensorMap tm_q;   // q       (D, Hq, T, B)                      box (64, G, T, 1)
  CUtensorMap tm_k;   // k_cache (128 B, slot, head, chunk, page)   box (128 B, BR, H2, NCH, 1)
  CUtensorMap tm_v;   // v_cache likewise
  CUtensorMap tm_ks;  // k_scratch (64, t, head, chunk, b)          box (64, TP, H2, NCH, 1)
  CUtensorMap tm_vs;  // v_scratch likewise
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;
  const float* v_scale;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  unsigned* unit_count;  // balanced schedule, combine fused into this kernel: arrivals per unit (else nullptr)
  int* err_flags;
  int B, T, Hq, Hkv, G, M, P, max_blocks, num_pages;
  int H2;          // kv heads per work unit
  int NHG;         // head groups per sequence, Hkv / H2
  int GT;          // query rows per kv head, G * T
  int TS;          // tokens per stage, 64 / H2
  int ilv;         // 1, 2 or 4: slice group ts takes only the stages j with j % ilv == ts % ilv
  int BR, lbr;     // rows of a page box, min(P, TS), and its log2
  int TP;          // scratch rows per box: T rounded up to a multiple of 8
  int num_splits;  // >= 1: explicit splits (grid = units x splits); 0: balanced (grid = CTAs)
  int tidar;       // 1: each sequence also attends to its T scratch tokens
  int draft_block; // draft token t sees scratch tokens [0, min(T, (t / draft_block + 1) * draft_block))
  int grid;        // CTAs of a balanced launch
  int item_w;      // balanced schedule: virtual pages charged for starting a work item on a unit
  float scale_log2;
};

struct ReduceParams {
  const float* part_o;
  const float* part_lse;
  __nv_bfloat16* out;
  float* lse;
  const int32_t* context_lens;
  int B, T, Hq, G, M, D, P, max_blocks, tidar;
  int H2, NHG, GT;
  int num_splits;  // >= 1: explicit layout [B][T][Hq][S]; 0: balanced-launch slots
  int grid;        // CTAs of the balanced split launch
  int item_w;      // the split launch's item_w
  int out_f16;     // 1: out holds f16 (else bf16)
};

// Shared-memory plan of one kernel instance (TSL: tokens per warp slice;
// CW: consumer warps, 4 or 8 -- with 8, two warps share each SM
// sub-partition and split each row tile's tokens).
template <int D, int MT, bool FP8, int TSL, int CW = kConsumerWarps>
struct Cfg {
  static constexpr bool REGSPLIT = CW == 8 && (FP8 || TSL >= 32);  // setmaxnreg layout (kSplitLaunchRegs)
  static constexpr int THREADS = 32 * (CW + (REGSPLIT ? 4 : 1));  // + the producer warp (warpgroup)
  static constexpr int ELEM = FP8 ? 1 : 2;
  static constexpr int CE = 128 / ELEM;         // elements per 128-byte row chunk
  static constexpr int NCH = D * ELEM / 128;    // row chunks per KV row
  static constexpr int SROWS = stage_rows(D * ELEM, FP8);
  static constexpr int TILE = SROWS * D * ELEM;  // bytes of the K (or V) tile of a stage
  static constexpr int STAGE = round_up(2 * TILE, 1024);
  static constexpr int ROWS = 16 * MT;
  static constexpr int QCH = D / 64;
  static constexpr int QCHUNK = ROWS * 128;
  static constexpr int QSLOT = QCH * QCHUNK;
  static constexpr int NGW = CW / MT;  // warps per row tile, each holding a partial result
  static constexpr int CHW = D <= 128 ? D : 64;    // output columns per merge round
  static constexpr int RSTR = CHW + 8;             // floats per row of the merge buffer
  static constexpr int RED = (NGW - 1) * ROWS * RSTR * 4;
  static constexpr int REDML = (NGW - 1) * ROWS * 2 * 4;
  static constexpr int BARS = 256;
  // fp8: per consumer warp a ring of kScaleRing handled stages' K and V
  // scales, one float per lane each.
  static constexpr int SRING = FP8 ? CW * kScaleRing * 2 * 32 * 4 : 0;
  static constexpr int FIXED = 2 * QSLOT + round_up(RED + REDML + SRING, 1024) + BARS;
  static constexpr int NS = clamp_int((kSmemBudget - FIXED) / STAGE, 2, 8);
  static constexpr int OFF_Q = NS * STAGE;
  static constexpr int OFF_RED = OFF_Q + 2 * QSLOT;
  static constexpr int OFF_REDML = OFF_RED + RED;
  static constexpr int OFF_SRING = OFF_REDML + REDML;
  static constexpr int OFF_BAR = round_up(OFF_SRING + SRING, 1024);
  static constexpr int OFF_PREFIX = OFF_BAR + BARS;
  static constexpr int SMEM_FIXED = OFF_PREFIX + 1024;  // + 1024 to align the dynamic base
  static_assert(D % 64 == 0 && (!FP8 || D >= 128), "unsupported head_dim");
  static_assert(MT == 1 || MT == 2 || MT == 4, "unsupported row tiles");
  static_assert(TSL == 16 || TSL == 32 || TSL == 64, "unsupported warp slice");
  // Fused combine: built into the instances whose main loop it costs no
  // spills (not fp8, not the register split); float4 column groups per
  // consumer thread and pass.
  static constexpr bool FUSED = !FP8 && !REGSPLIT;
  static constexpr int FEPT = clamp_int((ROWS * (D / 4) + 32 * CW - 1) / (32 * CW), 1, 4);
  static_assert(CW == 4 || CW == 8, "unsupported consumer warps");
  static_assert(2 * 8 + 6 <= BARS / 8, "barrier area: full/empty rings, Q slots, abort flag, fused-combine flag");
};

// ----------------------------------------------------------------- schedule
struct Item {
  int b, hg;          // sequence and head group (kv heads hg*H2 .. hg*H2+H2-1)
  int tok0, tok_end;  // paged tokens [tok0, tok_end) of sequence b
  int scratch;        // 1: the T draft-block scratch tokens follow (last stage)
  int nst;            // pipeline stages
  int part;           // -1: write the final out/lse; else the partial index
};

struct Cursor {
  long long f, f0, f1;  // balanced mode: this CTA's share of the flattened pages
  int done;             // explicit mode: the single item was handed out
};

__device__ __forceinline__ int clamp_ctx(const SplitParams& p, int c) {
  const int cap = p.max_blocks * p.P;
  return c < 0 ? 0 : (c > cap ? cap : c);
}

// Virtual pages of a (sequence, head group) unit in the balanced schedule:
// its pages and the draft-block scratch, plus item_w for the fixed cost of a
// work item on it (Q load, merge, partial write), so that a CTA whose share
// starts a unit takes that many fewer pages; none for a unit with no work.
__device__ __forceinline__ int unit_vpages(int ctx, int P, int tidar, int item_w) {
  const int v = (ctx + P - 1) / P + tidar;
  return v > 0 ? v + item_w : 0;
}

// a / b for a >= 0, b > 0: one 32-bit division while a fits in 32 bits (the
// usual case; the 64-bit division is a long software sequence on the path to
// a CTA's first page copy), the same quotient either way.
__device__ __forceinline__ long long div_nonneg(long long a, int b) {
  return a < (1LL << 32) ? (long long)((unsigned)a / (unsigned)b) : a / b;
}

__device__ __forceinline__ void cursor_init(const SplitParams& p, const int* s_start, Cursor& cur) {
  cur.done = 0;
  if (p.num_splits == 0) {
    const long long N = (long long)p.NHG * s_start[p.B];
    cur.f0 = div_nonneg(N * blockIdx.x, p.grid);
    cur.f1 = div_nonneg(N * (blockIdx.x + 1), p.grid);
    cur.f = cur.f0;
  }
}

// The next work item of this CTA; identical on every thread that calls it.
// Units are (sequence b, head group hg), u = b * NHG + hg.
__device__ __forceinline__ bool next_item(const SplitParams& p, const int* s_ctx, const int* s_start,
                                          Cursor& cur, Item& it) {
  const int P = p.P;
  if (p.num_splits > 0) {
    if (cur.done) return false;
    cur.done = 1;
    const int S = p.num_splits;
    const int s = blockIdx.y;
    const int u = blockIdx.x;
    it.b = u / p.NHG;
    it.hg = u % p.NHG;
    const int ctx = clamp_ctx(p, __ldg(p.context_lens + it.b));
    const int n = (ctx + P - 1) / P;
    const int pps = (n + S - 1) / S;
    const int p0 = min(n, s * pps);
    const int p1 = min(n, p0 + pps);
    it.tok0 = p0 * P;
    it.tok_end = max(it.tok0, min(p1 * P, ctx));
    it.scratch = (p.tidar && s == S - 1) ? 1 : 0;
    it.part = S == 1 ? -1 : s;
  } else {
    if (cur.f >= cur.f1) return false;
    const long long f = cur.f;
    const int NHG = p.NHG;
    int lo = 0, hi = p.B - 1;  // largest b with NHG * start[b] <= f (a non-empty sequence)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)NHG * s_start[mid] <= f) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int nv = s_start[b + 1] - s_start[b];
    const long long ub = (long long)NHG * s_start[b];
    const int hg = (int)div_nonneg(f - ub, nv);
    const long long us = ub + (long long)hg * nv;
    const long long ue = us + nv;
    const long long end = ue < cur.f1 ? ue : cur.f1;
    const int vp0 = (int)(f - us);
    const int vp1 = (int)(end - us);
    const int ctx = s_ctx[b];
    const int n = (ctx + P - 1) / P;
    // virtual pages [0, item_w) of the unit carry no keys; its pages follow
    const int rp0 = max(vp0 - p.item_w, 0), rp1 = max(vp1 - p.item_w, 0);
    it.b = b;
    it.hg = hg;
    it.tok0 = rp0 * P;
    it.tok_end = max(it.tok0, min(min(rp1, n) * P, ctx));
    it.scratch = (p.tidar && vp1 == nv) ? 1 : 0;  // the scratch is the unit's last virtual page
    it.part = (us >= cur.f0 && ue <= cur.f1) ? -1 : (b * NHG + hg + (int)blockIdx.x);
    cur.f = end;
  }
  it.nst = (it.tok_end - it.tok0 + p.TS - 1) / p.TS + it.scratch;
  return true;
}

// Swizzled byte offset of 16-byte unit `unit` in row `row` of a 128-byte-row
// tile whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int row, int unit) {
  return (uint32_t)(row * 128 + (((unit) ^ (row & 7)) << 4));
}

// Waits (bounded, ignoring the abort flag) for the last fill of every ring
// slot and Q slot this producer issued, so that no copy is still in flight
// when the CTA exits. `filled` has bit s set if slot s was ever filled, and
// `parity` holds the phase parity of its last fill; Q loads went to nq
// slots in turn.
__device__ __forceinline__ void drain_copies(uint32_t bar_full, uint32_t bar_qfull, int ns, uint32_t filled,
                                             uint32_t parity, int qloads, int nq = 2) {
  const int zero = 0;
  const volatile int* no_abort = &zero;
  for (int s = 0; s < ns; ++s)
    if (filled >> s & 1) mbar_wait(bar_full + 8 * s, parity >> s & 1, kWaitLimitNs, no_abort);
  for (int q = qloads - nq > 0 ? qloads - nq : 0; q < qloads; ++q)
    mbar_wait(bar_qfull + 8 * (q % nq), (q / nq) & 1, kWaitLimitNs, no_abort);
}

__device__ __forceinline__ void raise_abort(volatile int* s_abort, int* err_flags) {
  *s_abort = 1;
  atomicOr(err_flags, kErrWaitTimeout);
}

// Shared-memory ring that a producer warp fills: NS stages of `stage` bytes
// from sbase (each the K tile, then the V tile `tile` bytes further), and two
// Q slots of `qslot` bytes from sbase + off_q, each QCH column chunks of
// `qchunk` bytes. A stage tile is [page box][chunk][head][box row][128 B],
// or, with chunk_stride != 0 (one copy per page and chunk),
// [chunk][page box][head][box row][128 B] with chunks chunk_stride apart.
struct RingGeom {
  uint32_t sbase, off_q, qslot, qchunk, stage, tile;
  int ns, qch, nch;
  uint32_t row_bytes;     // bytes of one key row of all H2 heads
  uint32_t chunk_stride;  // 0: a box holds every chunk of its rows
  int nq;                 // Q slots (2: double-buffered across work items; 1)
};

// The tensor maps a launch copies through, fetched while the CTA's prologue
// (context lengths, prefix sums) runs, so that its first copies do not wait
// for their descriptors.
__device__ __forceinline__ void prefetch_maps(const SplitParams& p) {
  prefetch_tensormap(&p.tm_q);
  prefetch_tensormap(&p.tm_k);
  prefetch_tensormap(&p.tm_v);
  if (p.tidar) {
    prefetch_tensormap(&p.tm_ks);
    prefetch_tensormap(&p.tm_vs);
  }
}

// The producer warp of the split kernels: walks this CTA's work items and,
// per item, copies the Q rows of its H2 kv heads into a Q slot and every
// stage's K and V page boxes into the ring (one box per page, or the
// stage's rows of one page; the draft-token scratch as the last stage of
// its sequence's last item), after the consumers released the slot. Raises
// the abort flag on a timed-out wait and returns once every copy it issued
// has landed.
static __device__ __forceinline__ void produce_ring(const SplitParams& p, const int* s_ctx, const int* s_start,
                                                 const RingGeom& g, uint32_t bar_full, uint32_t bar_empty,
                                                 uint32_t bar_qfull, uint32_t bar_qempty, volatile int* s_abort,
                                                 int lane) {
  const uint32_t sbase = g.sbase;
  const int P = p.P;
  const int H2 = p.H2;
  const int TS = p.TS;
  const uint32_t row_bytes = g.row_bytes;
  const uint64_t pol_kv = l2_policy_evict_first();
  const uint64_t pol_q = l2_policy_evict_last();
  Cursor cur;
  cursor_init(p, s_start, cur);
  Item it;
  int stage = 0, qn = 0;
  uint32_t filled = 0, fill_parity = 0;
  bool ok = true;
  while (ok && next_item(p, s_ctx, s_start, cur, it)) {
    if (it.nst == 0) continue;
    // The item's block-table window is read first: the Q copies below
    // overlap its latency.
    const int32_t* bt_row = p.block_tables + (size_t)it.b * p.max_blocks;
    const int pbase = it.tok0 / P;
    const int npages = it.tok_end > it.tok0 ? (it.tok_end - 1) / P + 1 - pbase : 0;
    int ibase = 0;
    int ids = lane < npages ? __ldg(bt_row + pbase + lane) : 0;
    int ids_next = 32 + lane < npages ? __ldg(bt_row + pbase + 32 + lane) : 0;
    const int qs = qn % g.nq;
    // Warp-uniform verdicts: the lanes leave the loops together.
    if (qn >= g.nq)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_qempty + 8 * qs, ((qn / g.nq) - 1) & 1, kWaitLimitNs, s_abort));
    if (!ok) break;
    if (lane == 0) {
      // Rows of kv head hl occupy rows [hl*GT, (hl+1)*GT) of each chunk.
      const uint32_t qdst = sbase + g.off_q + qs * g.qslot;
      mbar_arrive_expect_tx(bar_qfull + 8 * qs, g.qch * p.M * 128);
      for (int hl = 0; hl < H2; ++hl)
#pragma unroll
        for (int c = 0; c < g.qch; ++c)
          tma_load_4d(qdst + c * g.qchunk + hl * p.GT * 128, &p.tm_q, bar_qfull + 8 * qs, c * 64,
                      (it.hg * H2 + hl) * p.G, 0, it.b, pol_q);
    }
    ++qn;

    for (int j = 0; j < it.nst; ++j, ++stage) {
      const int slot = stage % g.ns;
      if (stage >= g.ns) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_empty + 8 * slot, ((stage / g.ns) - 1) & 1, kWaitLimitNs, s_abort));
        if (!ok) break;
      }
      filled |= 1u << slot;
      fill_parity = (fill_parity & ~(1u << slot)) | (uint32_t((stage / g.ns) & 1) << slot);
      const uint32_t full = bar_full + 8 * slot;
      const uint32_t kdst = sbase + slot * g.stage;
      const uint32_t vdst = kdst + g.tile;
      const int ncb = g.chunk_stride ? g.nch : 1;  // copies per box: one per chunk, or one
      if (it.scratch && j == it.nst - 1) {
        if (lane == 0) {  // rows T..TP-1 of the box are outside the tensor: zero filled
          mbar_arrive_expect_tx(full, 2 * g.nch * H2 * p.TP * 128);
          for (int c = 0; c < ncb; ++c) {
            tma_load_5d(kdst + c * g.chunk_stride, &p.tm_ks, full, 0, 0, it.hg * H2, c, it.b, pol_kv);
            tma_load_5d(vdst + c * g.chunk_stride, &p.tm_vs, full, 0, 0, it.hg * H2, c, it.b, pol_kv);
          }
        }
        continue;
      }
      const int t_first = it.tok0 + j * TS;
      const int valid = min(TS, it.tok_end - t_first);
      const int pidx0 = t_first / P - pbase;  // page of the stage, relative to the item
      while (pidx0 >= ibase + 32) {           // advance the block-table window
        ibase += 32;
        ids = ids_next;
        ids_next = ibase + 32 + lane < npages ? __ldg(bt_row + pbase + ibase + 32 + lane) : 0;
      }
      if (P < TS) {  // whole pages: one box each
        const int npg = (valid + P - 1) / P;
        if (lane == 0) mbar_arrive_expect_tx(full, 2 * npg * P * row_bytes);
        for (int i = 0; i < npg; ++i) {
          const int page = __shfl_sync(0xffffffffu, ids, pidx0 - ibase + i);
          if (lane == 0) {
            const uint32_t boff = i * (g.chunk_stride ? 1 : g.nch) * H2 * P * 128;
            for (int c = 0; c < ncb; ++c) {
              tma_load_5d(kdst + c * g.chunk_stride + boff, &p.tm_k, full, 0, 0, it.hg * H2, c, page, pol_kv);
              tma_load_5d(vdst + c * g.chunk_stride + boff, &p.tm_v, full, 0, 0, it.hg * H2, c, page, pol_kv);
            }
          }
        }
      } else {  // TS rows of one page
        const int row0 = t_first % P;
        const int page = __shfl_sync(0xffffffffu, ids, pidx0 - ibase);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, 2 * TS * row_bytes);
          for (int c = 0; c < ncb; ++c) {
            tma_load_5d(kdst + c * g.chunk_stride, &p.tm_k, full, 0, row0, it.hg * H2, c, page, pol_kv);
            tma_load_5d(vdst + c * g.chunk_stride, &p.tm_v, full, 0, row0, it.hg * H2, c, page, pol_kv);
          }
        }
      }
    }
  }
  // Near the end of this CTA's work: the split-K reduce may be scheduled
  // (it waits for this grid to complete before reading any partial).
  launch_dependents();
  if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
  // Let every copy this warp issued land before the CTA can exit.
  drain_copies(bar_full, bar_qfull, g.ns, filled, fill_parity, qn, g.nq);
}

// ------------------------------------------------------- fused combine
// Pieces i0..i1 of the balanced schedule's unit u (the units' shares of the
// flattened pages meet inside it): CTA i wrote its piece to slot u + i,
// M rows of D floats and M lse values; a CTA whose share is empty wrote
// nothing. Source: the MSLK pull request "[ROCm] Add FlyDSL paged-attention
// decode backend (dense + fp8) with benchmark" (Kernels: the split-K partial
// combine), here run by the last CTA to finish a piece of the unit.
struct UnitPieces {
  int i0, i1;      // CTAs whose shares meet the unit
  long long N;     // flattened pages of the launch (all units)
};

__device__ __forceinline__ UnitPieces unit_pieces(const SplitParams& p, const int* s_start, const Item& it) {
  const long long nvb = s_start[it.b + 1] - s_start[it.b];
  UnitPieces r;
  r.N = (long long)p.NHG * s_start[p.B];
  const long long us = (long long)p.NHG * s_start[it.b] + (long long)it.hg * nvb;
  const long long ue = us + nvb;
  const long long G64 = p.grid;
  r.i0 = (int)(((us + 1) * G64 - 1) / r.N);
  r.i1 = (int)((ue * G64 - 1) / r.N);
  return r;
}

// Number of CTAs in [i0, i1] whose share holds at least one page.
__device__ __forceinline__ int written_pieces(const SplitParams& p, const UnitPieces& up) {
  const long long G64 = p.grid;
  if (up.N >= G64) return up.i1 - up.i0 + 1;
  int n = 0;
  for (long long i = up.i0; i <= up.i1; ++i) n += (up.N * i / G64) < (up.N * (i + 1) / G64);
  return n;
}

// Combines unit u's pieces into its final rows with nthr threads (index
// t): each thread takes float4 column groups (row rho, columns 4c..4c+3)
// of up to EPT of the unit's M x D/4 groups per pass and loads, for two
// pieces at a time, their lse and their columns of every group before
// combining (one online pass: running max, sums rescaled when it grows), so
// that a pass costs about one L2 round trip. Writes out (bf16, or f16 when
// F16) and, for column group 0 of a row, its lse; a NaN piece lse makes the
// row NaN, pieces with lse = -inf weigh 0.
// (Not inlined: its registers stay out of the split kernel's main loop.)
template <int D, bool F16, int EPT>
__device__ __noinline__ void fused_combine(const SplitParams& p, const Item& it, const UnitPieces& up, int t,
                                           int nthr) {
  constexpr int C4 = D / 4;
  constexpr int KG = 2;  // pieces per load round (EPT x KG float4 in flight per thread)
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float NaN = __int_as_float(0x7fffffff);
  const float LOG2E = 1.4426950408889634f;
  const int M = p.M, GT = p.GT, G = p.G;
  const int u = it.b * p.NHG + it.hg;
  const long long G64 = p.grid;
  const int np = up.i1 - up.i0 + 1;
  const int total = M * C4;
  for (int e0 = 0; e0 < total; e0 += EPT * nthr) {
    float m[EPT], L[EPT];
    float4 a[EPT];
    bool bad[EPT];
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
      m[q] = NEG_INF;
      L[q] = 0.f;
      a[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      bad[q] = false;
    }
    for (int k0 = 0; k0 < np; k0 += KG) {
      float lk[KG][EPT];
      float4 v[KG][EPT];
#pragma unroll
      for (int j = 0; j < KG; ++j) {
        const long long i = up.i0 + k0 + j;
        const bool in = k0 + j < np && (up.N >= G64 || (up.N * i / G64) < (up.N * (i + 1) / G64));
        const size_t slot = (size_t)(u + i);
#pragma unroll
        for (int q = 0; q < EPT; ++q) {
          const int e = e0 + q * nthr + t;
          const int rho = e / C4, c = e - rho * C4;
          const bool ok = in && e < total;
          lk[j][q] = ok ? __ldcg(p.part_lse + slot * M + rho) : NEG_INF;
          v[j][q] = ok ? __ldcg(reinterpret_cast<const float4*>(p.part_o + (slot * M + rho) * D) + c)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < EPT; ++q) {
        float mc = m[q];
#pragma unroll
        for (int j = 0; j < KG; ++j) {
          bad[q] |= lk[j][q] != lk[j][q];
          mc = fmaxf(mc, lk[j][q]);
        }
        if (mc == NEG_INF) continue;
        const float so = m[q] == NEG_INF ? 0.f : ex2((m[q] - mc) * LOG2E);
        a[q].x *= so; a[q].y *= so; a[q].z *= so; a[q].w *= so;
        L[q] *= so;
#pragma unroll
        for (int j = 0; j < KG; ++j) {
          if (lk[j][q] == NEG_INF) continue;
          const float w = ex2((lk[j][q] - mc) * LOG2E);
          a[q].x += w * v[j][q].x; a[q].y += w * v[j][q].y; a[q].z += w * v[j][q].z; a[q].w += w * v[j][q].w;
          L[q] += w;
        }
        m[q] = mc;
      }
    }
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
      const int e = e0 + q * nthr + t;
      if (e >= total) continue;
      const int rho = e / C4, c = e - rho * C4;
      // row rho = hl * GT + tq * G + j  ->  query head (hg * H2 + hl) * G + j
      const int hl = rho / GT, rem = rho - hl * GT;
      const int tq = rem / G;
      const size_t row = ((size_t)it.b * p.T + tq) * p.Hq + (size_t)(it.hg * p.H2 + hl) * G + (rem - tq * G);
      const float inv = bad[q] ? NaN : (L[q] > 0.f ? 1.f / L[q] : 0.f);
      *reinterpret_cast<uint2*>(p.out + row * D + 4 * c) =
          make_uint2(pack16<F16>(a[q].x * inv, a[q].y * inv), pack16<F16>(a[q].z * inv, a[q].w * inv));
      if (c == 0 && p.lse) p.lse[row] = bad[q] ? NaN : (L[q] > 0.f ? m[q] + lg2(L[q]) * kLn2 : NEG_INF);
    }
  }
}

// ------------------------------------------------------------ split kernel
// KV element kinds of the split kernel: bf16 (q, caches, out bf16), fp8
// (e4m3fn caches with scales; q and out bf16), f16 (q, caches, out f16).
constexpr int kKvBf16 = 0, kKvFp8 = 1, kKvF16 = 2;

template <int D, int MT, int KV, int TSL, int CW>
__global__ void __launch_bounds__(Cfg<D, MT, KV == kKvFp8, TSL, CW>::THREADS, 1)
    pa_split_kernel(const __grid_constant__ SplitParams p) {
  constexpr bool FP8 = KV == kKvFp8;
  constexpr bool F16 = KV == kKvF16;  // 16-bit path in f16 instead of bf16
  using C = Cfg<D, MT, FP8, TSL, CW>;
  constexpr int kThreads = C::THREADS;
  constexpr int NS = C::NS;
  constexpr int NGW = C::NGW;
  constexpr int NCH = C::NCH;
  constexpr int NTS = TSL / 8;  // n8 tiles of a warp's slice
  constexpr int NT8 = D / 8;    // n8 tiles of the output row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * NS;
  const uint32_t bar_qfull = bar_full + 16 * NS;
  const uint32_t bar_qempty = bar_qfull + 16;
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 2 * NS + 4);
  int* s_ctx = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
  int* s_start = s_ctx + (p.num_splits == 0 ? p.B : 0);

  if (tid == 32 * CW) prefetch_maps(p);  // the producer's lane 0
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, CW);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(bar_qfull + 8 * q, 1);
      mbar_init(bar_qempty + 8 * q, CW);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  // Query rows past M read as zero: clear both Q slots once.
  {
    uint4* q4 = reinterpret_cast<uint4*>(smem + C::OFF_Q);
    for (int i = tid; i < 2 * C::QSLOT / 16; i += kThreads) q4[i] = make_uint4(0, 0, 0, 0);
  }
  if (p.num_splits == 0) {
    for (int i = tid; i < p.B; i += kThreads) s_ctx[i] = clamp_ctx(p, __ldg(p.context_lens + i));
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
  __syncthreads();

  const int P = p.P;
  const int H2 = p.H2;
  const int TS = p.TS;
  // Bytes per key row of all H2 heads in a stage.
  const uint32_t row_bytes = H2 * D * C::ELEM;
  if (warp >= CW) {
    if constexpr (C::REGSPLIT) {
      regs_dec<kSplitProducerRegs>();
      if (warp != CW) return;  // the idle warps of the producer's warpgroup
    }
    const RingGeom g{sbase, (uint32_t)C::OFF_Q, (uint32_t)C::QSLOT, (uint32_t)C::QCHUNK, (uint32_t)C::STAGE,
                     (uint32_t)C::TILE, NS, C::QCH, NCH, row_bytes, 0u, 2};
    produce_ring(p, s_ctx, s_start, g, bar_full, bar_empty, bar_qfull, bar_qempty, s_abort, lane);
    return;
  }

  // ================================================================ consumers
  if constexpr (C::REGSPLIT) regs_inc<kSplitConsumerRegs>();
  // Warp w: row tile mt = w % MT; among the NGW warps of that tile, gi picks
  // the kv head hl (when a tile holds several heads' rows) and the token
  // slice ts of every stage (TSL tokens).
  const int GT = p.GT;
  const int mt = warp % MT;
  const int gi = warp / MT;
  const int hl_base = (mt * 16) / GT;
  const int ht = GT >= 16 ? 1 : max(1, min(16 / GT, H2 - hl_base));
  const int hl = min(hl_base + gi % ht, H2 - 1);  // (a tile of padding rows only reads head H2-1)
  const int ts = gi / ht;
  const int ph = ts % p.ilv;          // this warp's stages: j % ilv == ph
  const int tb = (ts / p.ilv) * TSL;  // first token of this warp's slice of a stage
  const int r = lane >> 2;
  const int c4 = lane & 3;
  const int rho0 = mt * 16 + r, rho1 = rho0 + 8;
  const bool rok0 = rho0 < p.M && rho0 / GT == hl;  // rows this warp computes
  const bool rok1 = rho1 < p.M && rho1 / GT == hl;
  // Scratch tokens the rows' draft tokens see (t = (rho % GT) / G): all T,
  // or the draft-block prefix of a block-masked draft.
  auto visible = [&](int rho) {
    const int t = (rho % GT) / p.G;
    return min(p.T, (t / p.draft_block + 1) * p.draft_block);
  };
  const int vis0 = visible(rho0), vis1 = visible(rho1);
  // Every row of this warp's tile is its own (draft units: G T >= 16): a
  // stage wholly inside the context then needs no score mask.
  const bool own_rows = __all_sync(0xffffffffu, rok0 && rok1);
  const int lp = 31 - __clz(p.P);  // log2 of the page size (a power of two)
  const uint64_t pol_scale = l2_policy_evict_first();
  const float NEG_INF = -__int_as_float(0x7f800000);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* redml = reinterpret_cast<float*>(smem + C::OFF_REDML);

  Cursor cur;
  cursor_init(p, s_start, cur);
  Item it;
  int stage = 0, qn = 0;
  bool ok = true;
  float acc[NT8][4];


  // Balanced schedule: a sequence with no keys has no work item; CTA
  // b % grid writes its rows (out = 0, lse = -inf).
  if (p.num_splits == 0 && !p.tidar) {
    const int ctid = warp * 32 + lane;
    for (int b = blockIdx.x; b < p.B; b += p.grid) {
      if (s_ctx[b] != 0) continue;
      const size_t rows = (size_t)p.T * p.Hq;
      uint4* o4 = reinterpret_cast<uint4*>(p.out + (size_t)b * rows * D);
      for (size_t i = ctid; i < rows * D / 8; i += 32 * CW) o4[i] = make_uint4(0, 0, 0, 0);
      if (p.lse)
        for (size_t i = ctid; i < rows; i += 32 * CW) p.lse[(size_t)b * rows + i] = NEG_INF;
    }
  }

  while (next_item(p, s_ctx, s_start, cur, it)) {
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    const int g = it.hg * H2 + hl;  // this warp's kv head

    if (it.nst > 0) {
      const int qs = qn & 1;
      const uint32_t qbase = sbase + C::OFF_Q + qs * C::QSLOT;
      if (ok) {
        ok = mbar_wait(bar_qfull + 8 * qs, (qn >> 1) & 1, kWaitLimitNs, s_abort);
        if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
      }
      if (FP8) {
        // Rewrite this item's Q rows, in place, as f16 A fragments whose k
        // order matches the fp8 K fragments: in k-step s, thread c4 holds
        // d = 16 s + 4 c4 .. +3. The fragments of k-steps 4q..4q+3 of row
        // tile mt take exactly the 2 KB that the tile's rows occupy in
        // column chunk q, so each chunk is converted by its own warp.
        if (gi == 0) {
          uint8_t* qs_ptr = smem + C::OFF_Q + qs * C::QSLOT;
          uint4* dst = reinterpret_cast<uint4*>(qs_ptr);
#pragma unroll
          for (int q = 0; q < D / 64; ++q) {
            uint32_t fr[4][4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int d = 16 * (4 * q + e) + 4 * c4;
#pragma unroll
              for (int h = 0; h < 2; ++h) {  // rows r and r + 8
                const int row = mt * 16 + r + 8 * h;
                uint2 v = make_uint2(0, 0);
                if (row < p.M)
                  v = *reinterpret_cast<const uint2*>(qs_ptr + q * C::QCHUNK + swz(row, (d % 64) / 8) + (d % 8) * 2);
                fr[e][h] = bf16x2_to_f16x2(v.x);
                fr[e][2 + h] = bf16x2_to_f16x2(v.y);
              }
            }
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[(q * C::QCHUNK + mt * 2048) / 16 + e * 32 + lane] = make_uint4(fr[e][0], fr[e][1], fr[e][2], fr[e][3]);
            __syncwarp();
          }
        }
        named_barrier_sync(1, 32 * CW);
      }
#pragma unroll
      for (int i = 0; i < NT8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

      // fp8 per-token scales, copied by the consumers themselves (small
      // copies per page through the tensor-copy engine cost more than the
      // K/V boxes they ride with): for the n-th stage this warp handles,
      // lane l copies the K and V scale of token tb + l % TSL into slot
      // n % kScaleRing of the warp's ring, kScaleAhead handled stages ahead,
      // by 4-byte asynchronous copies (one commit group per stage).
      const int32_t* bt_row = p.block_tables + (size_t)it.b * p.max_blocks;
      const int tok_l = it.tok0 + tb + (lane & (TSL - 1));  // this lane's token in stage 0
      const uint32_t ring = sbase + C::OFF_SRING + warp * (kScaleRing * 2 * 32 * 4);
      auto copy_scales = [&](int jj, int n) {  // stage jj, the warp's n-th handled stage
        const int tok = tok_l + jj * TS;
        if (tok < it.tok_end) {
          int pg = __ldg(bt_row + (tok >> lp));
          pg = (unsigned)pg < (unsigned)p.num_pages ? pg : 0;  // outside the pool: page 0's (finite) scales
          const size_t off = ((size_t)pg << lp | (tok & (P - 1))) * p.Hkv + g;
          const uint32_t dst = ring + (n % kScaleRing) * 256 + (lane & (TSL - 1)) * 4;
          if (lane < TSL) {
            cp_async4(dst, p.k_scale + off, pol_scale);
            cp_async4(dst + 128, p.v_scale + off, pol_scale);
          }
        }
        cp_async_commit();
      };
      int nh = 0;  // stages this warp handled in this item
      if (FP8) {
#pragma unroll
        for (int a = 0; a < kScaleAhead; ++a) copy_scales(ph + a * p.ilv, a);
      }

      for (int j = 0; j < it.nst; ++j) {
        const int st = stage + j;
        const int slot = st % NS;
        if (ok) {
          ok = mbar_wait(bar_full + 8 * slot, (st / NS) & 1, kWaitLimitNs, s_abort);
          if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
        }
        const bool scr = it.scratch && j == it.nst - 1;
        const int valid = scr ? p.T : min(TS, it.tok_end - (it.tok0 + j * TS));
        if (ok && tb < valid && ((j ^ ph) & (p.ilv - 1)) == 0) {
          // Stage tile: [box][chunk][head][box row][128 B]; a box holds the
          // rows of one page (scratch: TP rows). Every token index used below
          // is a multiple of 8 plus (lane & 7), so the 128-byte swizzle of its
          // row is (lane & 7) and only the row base depends on the token.
          const int lbt = scr ? 6 : p.lbr;
          const int brows = scr ? p.TP : p.BR;
          const uint32_t box_bytes = (uint32_t)(NCH * H2 * brows * 128);
          const uint32_t cstride = (uint32_t)(H2 * brows * 128);
          const uint32_t hoff = (uint32_t)(hl * brows * 128);
          auto row_base = [&](int tok) -> uint32_t {
            return (uint32_t)(tok >> lbt) * box_bytes + (uint32_t)(tok & ((1 << lbt) - 1)) * 128u + hoff;
          };
          const uint32_t kb_ = sbase + slot * C::STAGE;
          const uint32_t vb_ = kb_ + C::TILE;
          const int sw = lane & 7;
          const float* ksc = reinterpret_cast<const float*>(smem + C::OFF_SRING) +
                             warp * (kScaleRing * 2 * 32) + (nh % kScaleRing) * 64;  // [token - tb]
          const float* vsc = ksc + 32;
          if (FP8) {
            copy_scales(j + kScaleAhead * p.ilv, nh + kScaleAhead);
            cp_async_wait<kScaleAhead>();  // this stage's group has landed
            __syncwarp();                  // ... for every lane's copies
            ++nh;
          }

          // ---- S = Q K^T: 16 rows x TSL tokens. Slices of 16 tokens on
          // 16-bit pages: two accumulators per 8-token tile (even and odd
          // k-steps) halve the dependent MMA chain. Longer slices and fp8:
          // one (the slice's four or more tiles are the independent chains;
          // the registers go to the output).
          float s[NTS][4], s2[NTS][4];
#pragma unroll
          for (int i = 0; i < NTS; ++i) {
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
            s2[i][0] = s2[i][1] = s2[i][2] = s2[i][3] = 0.f;
          }
          if (!FP8) {
            uint32_t krow[NTS / 2];
#pragma unroll
            for (int nb = 0; nb < NTS / 2; ++nb) krow[nb] = kb_ + row_base(tb + nb * 16 + (lane >> 4) * 8 + sw);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              uint32_t qa[4];
              {
                const int row = mt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
                const int d = kk * 16 + (lane >> 4) * 8;
                ldsm_x4(qbase + (d / 64) * C::QCHUNK + swz(row, (d % 64) / 8), qa[0], qa[1], qa[2], qa[3]);
              }
              const int unit = ((kk * 16) % 64) / 8 + ((lane >> 3) & 1);
              const uint32_t coff = (kk / 4) * cstride + ((unit ^ sw) << 4);
#pragma unroll
              for (int nb = 0; nb < NTS / 2; ++nb) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(krow[nb] + coff, b0, b1, b2, b3);
                mma16<F16>((NTS <= 2 && (kk & 1)) ? s2[2 * nb] : s[2 * nb], qa, b0, b1);
                mma16<F16>((NTS <= 2 && (kk & 1)) ? s2[2 * nb + 1] : s[2 * nb + 1], qa, b2, b3);
              }
            }
          } else {
            uint32_t krow[NTS];
#pragma unroll
            for (int nt = 0; nt < NTS; ++nt) krow[nt] = kb_ + row_base(tb + nt * 8 + sw);
            const uint4* qf = reinterpret_cast<const uint4*>(smem + C::OFF_Q + qs * C::QSLOT);
#pragma unroll
            for (int kq = 0; kq < D / 64; ++kq) {
              uint32_t qa[4][4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint4 v = qf[(kq * C::QCHUNK + mt * 2048) / 16 + e * 32 + lane];
                qa[e][0] = v.x; qa[e][1] = v.y; qa[e][2] = v.z; qa[e][3] = v.w;
              }
              const int unit = 4 * kq + (lane >> 3);  // 16-byte unit = k-step
              const uint32_t coff = (unit / 8) * cstride + (((unit % 8) ^ sw) << 4);
              uint32_t kr[NTS][4];
#pragma unroll
              for (int nt = 0; nt < NTS; ++nt) ldsm_x4(krow[nt] + coff, kr[nt][0], kr[nt][1], kr[nt][2], kr[nt][3]);
              // Consecutive MMAs go to different score tiles: NTS independent
              // accumulation chains in flight instead of one.
#pragma unroll
              for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int nt = 0; nt < NTS; ++nt)
                  mma_f16(s[nt], qa[e], e4m3x2_to_f16x2(kr[nt][e]), e4m3x2_to_f16x2(kr[nt][e] >> 16));
            }
          }
#pragma unroll
          for (int i = 0; i < (FP8 || NTS > 2 ? 0 : NTS); ++i) {  // (only 16-token 16-bit slices use s2)
            s[i][0] += s2[i][0];
            s[i][1] += s2[i][1];
            s[i][2] += s2[i][2];
            s[i][3] += s2[i][3];
          }

          // ---- scale (and per-token K scale), mask, online softmax in base 2
          const float sl = p.scale_log2;
          if (!FP8 && own_rows && !scr && valid >= tb + TSL) {
#pragma unroll
            for (int i = 0; i < NTS; ++i) {
              s[i][0] *= sl;
              s[i][1] *= sl;
              s[i][2] *= sl;
              s[i][3] *= sl;
            }
          } else {
#pragma unroll
            for (int i = 0; i < NTS; ++i) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int tok = tb + i * 8 + 2 * c4 + (e & 1);
                float f = s[i][e] * sl;
                if (FP8) f *= ksc[tok - tb];
                const int lim = scr ? (e < 2 ? vis0 : vis1) : valid;
                s[i][e] = (tok < lim && (e < 2 ? rok0 : rok1)) ? f : NEG_INF;
              }
            }
          }
          float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
          for (int i = 0; i < NTS; ++i) {
            mx0 = fmaxf(mx0, fmaxf(s[i][0], s[i][1]));
            mx1 = fmaxf(mx1, fmaxf(s[i][2], s[i][3]));
          }
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
          constexpr float slack = FP8 ? 0.f : kMaxSlack;
          const float mn0 = mx0 > m0 + slack ? mx0 : m0, mn1 = mx1 > m1 + slack ? mx1 : m1;
          const float mu0 = mn0 == NEG_INF ? 0.f : mn0;
          const float mu1 = mn1 == NEG_INF ? 0.f : mn1;
          // alpha = 1 exactly when the running max did not move (also for
          // rows this warp does not compute, which stay at -inf).
          const float al0 = mn0 == m0 ? 1.f : ex2(m0 - mu0);
          const float al1 = mn1 == m1 ? 1.f : ex2(m1 - mu1);
          m0 = mn0;
          m1 = mn1;
          float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
          for (int i = 0; i < NTS; ++i) {
            s[i][0] = ex2(s[i][0] - mu0);
            s[i][1] = ex2(s[i][1] - mu0);
            s[i][2] = ex2(s[i][2] - mu1);
            s[i][3] = ex2(s[i][3] - mu1);
            ls0 += s[i][0] + s[i][1];
            ls1 += s[i][2] + s[i][3];
          }
          l0 = l0 * al0 + ls0;
          l1 = l1 * al1 + ls1;
          // The running max rarely moves after the first stages: rescale
          // the accumulator only when some row's max grew.
          if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < NT8; ++i) {
              acc[i][0] *= al0;
              acc[i][1] *= al0;
              acc[i][2] *= al1;
              acc[i][3] *= al1;
            }
          }

          // ---- O += P V: the score fragments are the A operand as they are
          const bool partial = valid < tb + TSL;
#pragma unroll
          for (int kb = 0; kb < NTS / 2; ++kb) {
            const int t0 = tb + kb * 16 + 2 * c4;  // tokens of the lo fragment; +8 for the hi one
            uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
            if (partial) {
              vm0 = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
              vm1 = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
            }
            const uint32_t vrow = vb_ + row_base(tb + kb * 16 + ((lane >> 3) & 1) * 8 + sw);
            uint32_t pa[4];
            if (!FP8) {
              pa[0] = pack16<F16>(s[2 * kb][0], s[2 * kb][1]);
              pa[1] = pack16<F16>(s[2 * kb][2], s[2 * kb][3]);
              pa[2] = pack16<F16>(s[2 * kb + 1][0], s[2 * kb + 1][1]);
              pa[3] = pack16<F16>(s[2 * kb + 1][2], s[2 * kb + 1][3]);
#pragma unroll
              for (int nd = 0; nd < D / 16; ++nd) {
                const int unit = ((nd * 16) % 64) / 8 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vrow + (nd / 4) * cstride + ((unit ^ sw) << 4), b0, b1, b2, b3);
                if (partial) {
                  b0 &= vm0; b1 &= vm1; b2 &= vm0; b3 &= vm1;
                }
                mma16<F16>(acc[2 * nd], pa, b0, b1);
                mma16<F16>(acc[2 * nd + 1], pa, b2, b3);
              }
            } else {
              // P~ = p * v_scale[token] in f16; masked tokens exactly 0.
              float vs[4];
              const int tl = kb * 16 + 2 * c4;  // t0 - tb
              vs[0] = t0 < valid ? vsc[tl] : 0.f;
              vs[1] = t0 + 1 < valid ? vsc[tl + 1] : 0.f;
              vs[2] = t0 + 8 < valid ? vsc[tl + 8] : 0.f;
              vs[3] = t0 + 9 < valid ? vsc[tl + 9] : 0.f;
              pa[0] = pack_f16x2(s[2 * kb][0] * vs[0], s[2 * kb][1] * vs[1]);
              pa[1] = pack_f16x2(s[2 * kb][2] * vs[0], s[2 * kb][3] * vs[1]);
              pa[2] = pack_f16x2(s[2 * kb + 1][0] * vs[2], s[2 * kb + 1][1] * vs[3]);
              pa[3] = pack_f16x2(s[2 * kb + 1][2] * vs[2], s[2 * kb + 1][3] * vs[3]);
#pragma unroll
              for (int uu = 0; uu < D / 32; ++uu) {
                const int unit = 2 * uu + (lane >> 4);
                uint32_t R[4];
                ldsm_x4_trans(vrow + (unit / 8) * cstride + (((unit % 8) ^ sw) << 4), R[0], R[1], R[2], R[3]);
                if (partial) {
                  R[0] &= vm0; R[1] &= vm1; R[2] &= vm0; R[3] &= vm1;
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                  // bytes (tok 2c d 2r, tok 2c d 2r+1, tok 2c+1 d 2r, tok 2c+1 d 2r+1)
                  const uint32_t x = prmt(R[2 * k], 0, 0x3120);
                  const uint32_t y = prmt(R[2 * k + 1], 0, 0x3120);
                  const int nt = 2 * (2 * uu + k);
                  mma_f16(acc[nt], pa, e4m3x2_to_f16x2(x), e4m3x2_to_f16x2(y));
                  mma_f16(acc[nt + 1], pa, e4m3x2_to_f16x2(x >> 16), e4m3x2_to_f16x2(y >> 16));
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
      }
      stage += it.nst;
      if (FP8) fence_proxy_async_smem();  // the slot was rewritten through the generic proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_qempty + 8 * qs);
      ++qn;
    } else {
#pragma unroll
      for (int i = 0; i < NT8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    }

    // ---- merge the NGW warps of each row tile, then write
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    // Rounds of CHW output columns: the other warps of the tile write their
    // columns (and, in the first round, their m and l), warp gi = 0 folds
    // them into its own, each weighted by 2^(m_warp - M) / L.
    float M0 = m0, M1 = m1, L0 = 0.f, L1 = 0.f, w00 = 1.f, w01 = 1.f, inv0 = 0.f, inv1 = 0.f;
    float wq0[NGW > 1 ? NGW - 1 : 1], wq1[NGW > 1 ? NGW - 1 : 1];
    auto merge_weights = [&]() {
#pragma unroll
      for (int q = 0; q < NGW - 1; ++q) {
        M0 = fmaxf(M0, redml[(q * C::ROWS + rho0) * 2]);
        M1 = fmaxf(M1, redml[(q * C::ROWS + rho1) * 2]);
      }
      const float Mu0 = M0 == NEG_INF ? 0.f : M0;
      const float Mu1 = M1 == NEG_INF ? 0.f : M1;
      w00 = ex2(m0 - Mu0);
      w01 = ex2(m1 - Mu1);
      L0 = w00 * l0;
      L1 = w01 * l1;
#pragma unroll
      for (int q = 0; q < NGW - 1; ++q) {
        wq0[q] = ex2(redml[(q * C::ROWS + rho0) * 2] - Mu0);
        wq1[q] = ex2(redml[(q * C::ROWS + rho1) * 2] - Mu1);
        L0 += wq0[q] * redml[(q * C::ROWS + rho0) * 2 + 1];
        L1 += wq1[q] * redml[(q * C::ROWS + rho1) * 2 + 1];
      }
      inv0 = L0 > 0.f ? 1.f / L0 : 0.f;
      inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    };
    auto merge_columns = [&](int i0, int i1) {  // n8 tiles [i0, i1) of this round
#pragma unroll
      for (int i = i0; i < i1; ++i) {
        float a0 = acc[i][0] * w00, a1 = acc[i][1] * w00, a2 = acc[i][2] * w01, a3 = acc[i][3] * w01;
#pragma unroll
        for (int q = 0; q < NGW - 1; ++q) {
          const float* rb = red + (size_t)q * C::ROWS * C::RSTR + (i - i0) * 8 + 2 * c4;
          const float2 x = *reinterpret_cast<const float2*>(rb + rho0 * C::RSTR);
          const float2 y = *reinterpret_cast<const float2*>(rb + rho1 * C::RSTR);
          a0 += wq0[q] * x.x;
          a1 += wq0[q] * x.y;
          a2 += wq1[q] * y.x;
          a3 += wq1[q] * y.y;
        }
        acc[i][0] = a0 * inv0;
        acc[i][1] = a1 * inv0;
        acc[i][2] = a2 * inv1;
        acc[i][3] = a3 * inv1;
      }
    };
    if constexpr (NGW > 1) {
#pragma unroll
      for (int ck = 0; ck < D / C::CHW; ++ck) {
        constexpr int NCT = C::CHW / 8;  // n8 tiles per round
        named_barrier_sync(1, 32 * CW);  // the previous round's (or item's) reads are done
        if (gi > 0) {
          float* rb = red + (size_t)(gi - 1) * C::ROWS * C::RSTR;
#pragma unroll
          for (int i = 0; i < NCT; ++i) {
            const int ia = ck * NCT + i;
            *reinterpret_cast<float2*>(rb + rho0 * C::RSTR + i * 8 + 2 * c4) = make_float2(acc[ia][0], acc[ia][1]);
            *reinterpret_cast<float2*>(rb + rho1 * C::RSTR + i * 8 + 2 * c4) = make_float2(acc[ia][2], acc[ia][3]);
          }
          if (ck == 0 && c4 == 0) {
            float* ml = redml + (size_t)(gi - 1) * C::ROWS * 2;
            ml[2 * rho0] = m0;
            ml[2 * rho0 + 1] = l0;
            ml[2 * rho1] = m1;
            ml[2 * rho1 + 1] = l1;
          }
        }
        named_barrier_sync(1, 32 * CW);
        if (gi == 0) {
          if (ck == 0) merge_weights();
          merge_columns(ck * NCT, (ck + 1) * NCT);
        }
      }
    } else {
      merge_weights();
      merge_columns(0, NT8);
    }
    // Combine fused into this kernel (balanced schedule; instances with
    // C::FUSED): every warp takes part in the arrival below, the tile's
    // first warp writes the piece.
    const bool fused = C::FUSED && p.unit_count != nullptr && it.part >= 0;
    if (gi != 0 && !fused) continue;
    if (gi == 0) {
      float lse0 = L0 > 0.f ? (M0 + lg2(L0)) * kLn2 : NEG_INF;
      float lse1 = L1 > 0.f ? (M1 + lg2(L1)) * kLn2 : NEG_INF;
      // An item cut short by a timed-out wait (in this warp or another role of
      // the CTA) is written as NaN, so that no part of it passes as a result.
      if (__any_sync(0xffffffffu, !ok || *s_abort)) {
        const float NaN = __int_as_float(0x7fffffff);
  #pragma unroll
        for (int i = 0; i < NT8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = NaN;
        lse0 = lse1 = NaN;
      }

  #pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int rho = h2 ? rho1 : rho0;
        if (rho >= p.M) continue;
        // row rho = hl * GT + t * G + j  ->  query head (hg * H2 + hl) * G + j
        const int rhl = rho / GT, rem = rho - rhl * GT;
        const int t = rem / p.G;
        const int h = (it.hg * H2 + rhl) * p.G + (rem - t * p.G);
        const size_t row = ((size_t)it.b * p.T + t) * p.Hq + h;
        const float lsev = h2 ? lse1 : lse0;
        if (it.part < 0) {
          __nv_bfloat16* o = p.out + row * D;
          if (!FP8) {
  #pragma unroll
            for (int i = 0; i < NT8; ++i)
              *reinterpret_cast<uint32_t*>(o + i * 8 + 2 * c4) = pack16<F16>(acc[i][2 * h2], acc[i][2 * h2 + 1]);
          } else {
  #pragma unroll
            for (int u = 0; u < D / 16; ++u)
              *reinterpret_cast<uint2*>(o + 16 * u + 4 * c4) =
                  make_uint2(pack_bf16x2(acc[2 * u][2 * h2], acc[2 * u + 1][2 * h2]),
                             pack_bf16x2(acc[2 * u][2 * h2 + 1], acc[2 * u + 1][2 * h2 + 1]));
          }
          if (c4 == 0 && p.lse) p.lse[row] = lsev;
        } else {
          const size_t prow = p.num_splits > 0 ? row * p.num_splits + it.part : (size_t)it.part * p.M + rho;
          float* o = p.part_o + prow * D;
          if (!FP8) {
  #pragma unroll
            for (int i = 0; i < NT8; ++i)
              *reinterpret_cast<float2*>(o + i * 8 + 2 * c4) = make_float2(acc[i][2 * h2], acc[i][2 * h2 + 1]);
          } else {
  #pragma unroll
            for (int u = 0; u < D / 16; ++u)
              *reinterpret_cast<float4*>(o + 16 * u + 4 * c4) =
                  make_float4(acc[2 * u][2 * h2], acc[2 * u + 1][2 * h2], acc[2 * u][2 * h2 + 1],
                              acc[2 * u + 1][2 * h2 + 1]);
          }
          if (c4 == 0) p.part_lse[prow] = lsev;
        }
      }
    }
    if constexpr (C::FUSED) {
      if (fused) {
        // The last CTA to finish a piece of this unit combines all of them:
        // each piece's rows are made visible device-wide before its CTA
        // counts itself in (atomicInc wraps to 0 on the last arrival, so the
        // counters are zero again after every unit), and the last CTA reads
        // the other pieces only after its own arrival.
        volatile unsigned* s_last = reinterpret_cast<volatile unsigned*>(bars + 2 * NS + 5);
        __threadfence();
        named_barrier_sync(1, 32 * CW);
        const UnitPieces up = unit_pieces(p, s_start, it);
        if (warp == 0 && lane == 0) {
          const unsigned np = (unsigned)written_pieces(p, up);
          const unsigned old = atomicInc(p.unit_count + it.b * p.NHG + it.hg, np - 1);
          *s_last = old == np - 1 ? 1u : 0u;
        }
        named_barrier_sync(1, 32 * CW);
        if (*s_last) {
          __threadfence();
          fused_combine<D, F16, C::FEPT>(p, it, up, warp * 32 + lane, 32 * CW);
        }
        named_barrier_sync(1, 32 * CW);  // s_last is read before the next arrival rewrites it
      }
    }
  }
  if (FP8) cp_async_wait<0>();  // no scale copy may still be landing when the CTA exits
  launch_dependents();
}

}  // namespace pa
