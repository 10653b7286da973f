// Split kernel with paired consumer roles (included by the instance units).
//
// Same operation, schedule, ring, partials and outputs as pa_split_kernel
// (pa_kernels.cuh), with each consumer's per-stage chain split between
// three warps. Sources:
// the MSLK pull request "[ROCm] Add FlyDSL paged-attention decode backend
// (dense + fp8) with benchmark" (Kernels: head-packed matrix-core decode,
// native fp8 e4m3fn KV with symmetric per-token scale, split-K partials) and
// the ROCm blog page "Implementing a High-Performance Custom Diffusion
// Attention Kernel with FlyDSL" ("Match MFMA Operands to the Desired
// Fragment Layout"; "Prefetch Data").
//
// GB300 design. In the single-role kernel one warp per SM sub-partition
// runs ldmatrix -> (fp8: e4m3 -> f16) -> Q K^T MMAs -> softmax -> P V MMAs
// for every stage, and with nothing else to issue on its sub-partition the
// fixed latencies of that chain are exposed. Here every (row tile, slice
// group) pair owns three warps on one sub-partition: the S warp (warps 0-3)
// computes the scores, the online max and sum and the P operand (fp8: times
// the per-token V scale) and sends P with the rows' rescale factors to two
// PV warps (warps 4-7: output columns [0, D/2); warps 8-11: [D/2, D))
// through a message slot in shared memory (mbarriers; all lanes arrive,
// every wait bounded; the S warp runs up to one slice ahead); each PV warp
// holds its half of the output
// accumulator, rescales it, runs P V on its half of the stage's value
// columns and releases the stage. The three chains overlap across stages.
// Closing a work item the S warp sends its running max and sum, and the PV
// warps of a row tile merge and write their columns as the single-role
// kernel does. Warpgroup 3 holds the producer (produce_ring) and three idle
// warps; setmaxnreg moves their registers to the three consumer warpgroups
// (kPair* constants).
#pragma once

#include "pa_kernels.cuh"

namespace pa {

// Registers per thread: 128 at launch (16 warps); the producer's warpgroup
// drops to 40 and the three consumer warpgroups rise to 152:
// 3 x 128 x 152 + 128 x 40 <= 512 x 128.
constexpr int kPairLaunchRegs = 128, kPairConsumerRegs = 152, kPairProducerRegs = 40;
// Shared memory for the ring and fixed areas (the opt-in maximum is 227 KB).
// A work item's stages stay in the ring from the S warps' use until the PV
// warps' (an S warp runs up to one slice ahead), so the ring takes every
// byte the fixed areas leave: one Q slot, one message slot per pair and
// 16-column merge rounds.
constexpr int kPairSmemBudget = 226 * 1024;
static_assert(3 * 128 * kPairConsumerRegs + 128 * kPairProducerRegs <= 512 * kPairLaunchRegs,
              "register split exceeds the launch pool");

template <int D, int MT, bool FP8, int TSL>
struct PCfg {
  static constexpr int PAIRS = 4;                 // (row tile, slice group) pairs: one per SM sub-partition
  static constexpr int THREADS = 512;              // S warps, two PV warps per pair, the producer's warpgroup
  static constexpr int DH = D / 2;                // output columns of a PV warp
  static constexpr int ELEM = FP8 ? 1 : 2;
  static constexpr int NCH = D * ELEM / 128;
  static constexpr int SROWS = stage_rows(D * ELEM, FP8);
  static constexpr int TILE = SROWS * D * ELEM;
  static constexpr int STAGE = round_up(2 * TILE, 1024);
  static constexpr int ROWS = 16 * MT;
  static constexpr int QCH = D / 64;
  static constexpr int QCHUNK = ROWS * 128;
  static constexpr int QSLOT = QCH * QCHUNK;
  static constexpr int NQ = 1;  // Q slots
  static constexpr int NGW = PAIRS / MT;  // pairs per row tile, each holding a partial result
  static constexpr int CHW = 16;  // output columns per merge round (of a PV warp's half)
  static constexpr int RSTR = CHW + 8;
  static constexpr int RED = 2 * (NGW - 1) * ROWS * RSTR * 4;
  static constexpr int REDML = (NGW - 1) * ROWS * 2 * 4;
  static constexpr int SRING = FP8 ? PAIRS * kScaleRing * 2 * 32 * 4 : 0;
  // A message: the P fragments of one slice (TSL / 4 words per lane), then
  // the rows' rescale factors (closing an item: m0, m1, l0, l1), stored as
  // [uint4 group][lane].
  static constexpr int NPW = TSL / 4;
  static constexpr int MSGV = NPW / 4 + 1;
  static constexpr int MSG = MSGV * 32 * 16;
  static constexpr int NMSG = 1;  // message slots per pair
  static constexpr int PMSG = PAIRS * NMSG * MSG;
  static constexpr int BARS = 512;
  static constexpr int FIXED = NQ * QSLOT + round_up(RED + REDML + SRING + PMSG, 1024) + BARS;
  static constexpr int NS = clamp_int((kPairSmemBudget - FIXED) / STAGE, 2, 8);
  static constexpr int OFF_Q = NS * STAGE;
  static constexpr int OFF_RED = OFF_Q + NQ * QSLOT;
  static constexpr int OFF_REDML = OFF_RED + RED;
  static constexpr int OFF_SRING = OFF_REDML + REDML;
  static constexpr int OFF_PMSG = OFF_SRING + SRING;
  static constexpr int OFF_BAR = round_up(OFF_PMSG + PMSG, 1024);
  static constexpr int OFF_PREFIX = OFF_BAR + BARS;
  static constexpr int SMEM_FIXED = OFF_PREFIX + 1024;
  static_assert(D % 64 == 0 && (!FP8 || D >= 128), "unsupported head_dim");
  static_assert(MT == 1 || MT == 2 || MT == 4, "unsupported row tiles");
  static_assert(TSL == 16 || TSL == 32 || TSL == 64, "unsupported warp slice");
  static_assert(DH % CHW == 0, "merge rounds");
  static_assert((2 * 8 + 5 + 2 * PAIRS * NMSG) * 8 <= BARS, "barrier area");
};

template <int D, int MT, int KV, int TSL>
__global__ void __launch_bounds__(PCfg<D, MT, KV == kKvFp8, TSL>::THREADS, 1)
    pa_pair_kernel(const __grid_constant__ SplitParams p) {
  constexpr bool FP8 = KV == kKvFp8;
  constexpr bool F16 = KV == kKvF16;
  using C = PCfg<D, MT, FP8, TSL>;
  constexpr int NS = C::NS;
  constexpr int NGW = C::NGW;
  constexpr int NCH = C::NCH;
  constexpr int PAIRS = C::PAIRS;
  constexpr int NMSG = C::NMSG;
  constexpr int NTS = TSL / 8;  // n8 tiles of a warp's slice
  constexpr int NT8 = C::DH / 8;  // n8 tiles of a PV warp's output columns
  constexpr int DH = C::DH;
  constexpr int NPW = C::NPW;
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
  const uint32_t bar_pfull = bar_full + 8 * (2 * NS + 5);     // [pair][slot]
  const uint32_t bar_pempty = bar_pfull + 8 * PAIRS * NMSG;  // [pair][slot]
  int* s_ctx = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
  int* s_start = s_ctx + (p.num_splits == 0 ? p.B : 0);

  if (tid == 32 * 3 * PAIRS) prefetch_maps(p);  // the producer's lane 0
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 2 * PAIRS);  // the PV warps
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(bar_qfull + 8 * q, 1);
      mbar_init(bar_qempty + 8 * q, PAIRS);  // the S warps
    }
    for (int i = 0; i < PAIRS * NMSG; ++i) {
      mbar_init(bar_pfull + 8 * i, 32);       // the S warp's lanes
      mbar_init(bar_pempty + 8 * i, 64);      // both PV warps' lanes
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  // Query rows past M read as zero: clear both Q slots once.
  {
    uint4* q4 = reinterpret_cast<uint4*>(smem + C::OFF_Q);
    for (int i = tid; i < C::NQ * C::QSLOT / 16; i += C::THREADS) q4[i] = make_uint4(0, 0, 0, 0);
  }
  if (p.num_splits == 0) {
    for (int i = tid; i < p.B; i += C::THREADS) s_ctx[i] = clamp_ctx(p, __ldg(p.context_lens + i));
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

  const int H2 = p.H2;
  const int TS = p.TS;
  const uint32_t row_bytes = H2 * D * C::ELEM;
  if (warp >= 3 * PAIRS) {
    regs_dec<kPairProducerRegs>();
    if (warp != 3 * PAIRS) return;  // the idle warps of the producer's warpgroup
    const RingGeom g{sbase, (uint32_t)C::OFF_Q, (uint32_t)C::QSLOT, (uint32_t)C::QCHUNK, (uint32_t)C::STAGE,
                     (uint32_t)C::TILE, NS, C::QCH, NCH, row_bytes, 0u, C::NQ};
    produce_ring(p, s_ctx, s_start, g, bar_full, bar_empty, bar_qfull, bar_qempty, s_abort, lane);
    return;
  }

  // ================================================================ consumers
  regs_inc<kPairConsumerRegs>();
  const bool s_role = warp < PAIRS;
  const int cw = warp & (PAIRS - 1);  // the pair
  const int hh = warp >= 2 * PAIRS ? 1 : 0;  // PV warps: half of the output columns
  // Pair cw: row tile mt = cw % MT; among the NGW pairs of that tile, gi
  // picks the kv head hl (when a tile holds several heads' rows) and the
  // token slice ts of every stage (TSL tokens).
  const int GT = p.GT;
  const int mt = cw % MT;
  const int gi = cw / MT;
  const int hl_base = (mt * 16) / GT;
  const int ht = GT >= 16 ? 1 : max(1, min(16 / GT, H2 - hl_base));
  const int hl = min(hl_base + gi % ht, H2 - 1);
  const int ts = gi / ht;
  const int ph = ts % p.ilv;
  const int tb = (ts / p.ilv) * TSL;
  const int r = lane >> 2;
  const int c4 = lane & 3;
  const int rho0 = mt * 16 + r, rho1 = rho0 + 8;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int lp = 31 - __clz(p.P);
  uint4* msg_base = reinterpret_cast<uint4*>(smem + C::OFF_PMSG) + cw * NMSG * (C::MSG / 16) + lane;
  int nmsg = 0;  // messages of this pair so far (sent by its S warp, taken by its PV warp)

  Cursor cur;
  cursor_init(p, s_start, cur);
  Item it{};
  int stage = 0, qn = 0;
  bool ok = true;

  // Stage j of the current item: its valid tokens, and whether this pair
  // takes a slice of it (the same verdict on both warps of the pair).
  auto stage_valid = [&](int j) {
    const bool scr = it.scratch && j == it.nst - 1;
    return scr ? p.T : min(TS, it.tok_end - (it.tok0 + j * TS));
  };
  auto handled = [&](int j) { return tb < stage_valid(j) && ((j ^ ph) & (p.ilv - 1)) == 0; };

  if (s_role) {
    // ============================================================ S warps
    const bool rok0 = rho0 < p.M && rho0 / GT == hl;
    const bool rok1 = rho1 < p.M && rho1 / GT == hl;
    auto visible = [&](int rho) {
      const int t = (rho % GT) / p.G;
      return min(p.T, (t / p.draft_block + 1) * p.draft_block);
    };
    const int vis0 = visible(rho0), vis1 = visible(rho1);
    const uint64_t pol_scale = l2_policy_evict_first();
    // Sends one message: NPW P words, then two more floats (and two spare).
    auto send = [&](const uint32_t* words, float a, float b, float c, float d) {
      const int ms = nmsg % NMSG;
      if (nmsg >= NMSG && ok) {
        ok = mbar_wait(bar_pempty + 8 * (cw * NMSG + ms), ((nmsg / NMSG) - 1) & 1, kWaitLimitNs, s_abort);
        if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
      }
      uint4* m = msg_base + ms * (C::MSG / 16);
#pragma unroll
      for (int v = 0; v < NPW / 4; ++v)
        m[v * 32] = make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]);
      m[(NPW / 4) * 32] = make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c), __float_as_uint(d));
      mbar_arrive(bar_pfull + 8 * (cw * NMSG + ms));
      ++nmsg;
    };

    while (next_item(p, s_ctx, s_start, cur, it)) {
      float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
      const int g = it.hg * H2 + hl;  // this pair's kv head
      if (it.nst > 0) {
        const int qs = qn % C::NQ;
        const uint32_t qbase = sbase + C::OFF_Q + qs * C::QSLOT;
        if (ok) {
          ok = mbar_wait(bar_qfull + 8 * qs, (qn / C::NQ) & 1, kWaitLimitNs, s_abort);
          if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
        }
        if (FP8) {
          // Q rows rewritten in place as f16 A fragments whose k order
          // matches the e4m3 K fragments (as in the single-role kernel).
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
                for (int h = 0; h < 2; ++h) {
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
          named_barrier_sync(1, 32 * PAIRS);
        }
        // fp8 per-token scales: copied by the S warp itself a few handled
        // stages ahead into its ring (as in the single-role kernel).
        const int32_t* bt_row = p.block_tables + (size_t)it.b * p.max_blocks;
        const int tok_l = it.tok0 + tb + (lane & (TSL - 1));
        const uint32_t ring = sbase + C::OFF_SRING + cw * (kScaleRing * 2 * 32 * 4);
        // The page of this lane's token in stage jj (loaded one handled stage
        // before its scale copy, off the copy's dependency chain).
        auto page_of = [&](int jj) -> int {
          const int tok = tok_l + jj * TS;
          return tok < it.tok_end ? __ldg(bt_row + (tok >> lp)) : 0;
        };
        auto copy_scales = [&](int jj, int n, int pg) {  // pg: page_of(jj)
          const int tok = tok_l + jj * TS;
          if (tok < it.tok_end) {
            pg = (unsigned)pg < (unsigned)p.num_pages ? pg : 0;
            const size_t off = ((size_t)pg << lp | (tok & (p.P - 1))) * p.Hkv + g;
            const uint32_t dst = ring + (n % kScaleRing) * 256 + (lane & (TSL - 1)) * 4;
            if (lane < TSL) {
              cp_async4(dst, p.k_scale + off, pol_scale);
              cp_async4(dst + 128, p.v_scale + off, pol_scale);
            }
          }
          cp_async_commit();
        };
        int nh = 0;
        int pg_next = 0;  // page_of() of the next scale copy
        if (FP8) {
#pragma unroll
          for (int a = 0; a < kScaleAhead; ++a) copy_scales(ph + a * p.ilv, a, page_of(ph + a * p.ilv));
          pg_next = page_of(ph + kScaleAhead * p.ilv);
        }

        for (int j = 0; j < it.nst; ++j) {
          if (!handled(j)) continue;
          const int st = stage + j;
          const int slot = st % NS;
          if (ok) {
            ok = mbar_wait(bar_full + 8 * slot, (st / NS) & 1, kWaitLimitNs, s_abort);
            if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
          }
          const bool scr = it.scratch && j == it.nst - 1;
          const int valid = stage_valid(j);
          uint32_t pw[NPW];
          float al0 = 1.f, al1 = 1.f;
#pragma unroll
          for (int i = 0; i < NPW; ++i) pw[i] = 0u;
          if (FP8) {
            copy_scales(j + kScaleAhead * p.ilv, nh + kScaleAhead, pg_next);
            pg_next = page_of(j + (kScaleAhead + 1) * p.ilv);
            cp_async_wait<kScaleAhead>();
            __syncwarp();
          }
          const float* ksc = reinterpret_cast<const float*>(smem + C::OFF_SRING) + cw * (kScaleRing * 2 * 32) +
                             (nh % kScaleRing) * 64;
          const float* vsc = ksc + 32;
          if (FP8) ++nh;
          if (ok) {
            const int lbt = scr ? 6 : p.lbr;
            const int brows = scr ? p.TP : p.BR;
            const uint32_t box_bytes = (uint32_t)(NCH * H2 * brows * 128);
            const uint32_t cstride = (uint32_t)(H2 * brows * 128);
            const uint32_t hoff = (uint32_t)(hl * brows * 128);
            auto row_base = [&](int tok) -> uint32_t {
              return (uint32_t)(tok >> lbt) * box_bytes + (uint32_t)(tok & ((1 << lbt) - 1)) * 128u + hoff;
            };
            const uint32_t kb_ = sbase + slot * C::STAGE;
            const int sw = lane & 7;

            // ---- S = Q K^T: 16 rows x TSL tokens, one accumulator per tile
            float s[NTS][4];
#pragma unroll
            for (int i = 0; i < NTS; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
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
                  mma16<F16>(s[2 * nb], qa, b0, b1);
                  mma16<F16>(s[2 * nb + 1], qa, b2, b3);
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
                const int unit = 4 * kq + (lane >> 3);
                const uint32_t coff = (unit / 8) * cstride + (((unit % 8) ^ sw) << 4);
                uint32_t kr[NTS][4];
#pragma unroll
                for (int nt = 0; nt < NTS; ++nt) ldsm_x4(krow[nt] + coff, kr[nt][0], kr[nt][1], kr[nt][2], kr[nt][3]);
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                  for (int nt = 0; nt < NTS; ++nt)
                    mma_f16(s[nt], qa[e], e4m3x2_to_f16x2(kr[nt][e]), e4m3x2_to_f16x2(kr[nt][e] >> 16));
              }
            }

            // ---- scale (and per-token K scale), mask, online softmax in base 2
            const float sl = p.scale_log2;
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
            // fp8: P~ = p * v_scale is f16, so the running max may lag by
            // kMaxSlack (p <= 2^8) only while every v_scale of the slice is
            // below 2^7 (P~ < 2^15); else it tracks the exact max.
            float slack = kMaxSlack;
            if (FP8) {
              const uint32_t vb = (lane < TSL && tb + lane < valid) ? __float_as_uint(fabsf(vsc[lane])) : 0u;
              slack = __reduce_max_sync(0xffffffffu, vb) < 0x43000000u ? kMaxSlack : 0.f;  // 128.0f
            }
            const float mn0 = mx0 > m0 + slack ? mx0 : m0, mn1 = mx1 > m1 + slack ? mx1 : m1;
            const float mu0 = mn0 == NEG_INF ? 0.f : mn0;
            const float mu1 = mn1 == NEG_INF ? 0.f : mn1;
            al0 = mn0 == m0 ? 1.f : ex2(m0 - mu0);
            al1 = mn1 == m1 ? 1.f : ex2(m1 - mu1);
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

            // ---- the P operand (16-bit; fp8: p * v_scale[token] in f16,
            // masked tokens exactly 0)
#pragma unroll
            for (int kb = 0; kb < NTS / 2; ++kb) {
              if (!FP8) {
                pw[4 * kb] = pack16<F16>(s[2 * kb][0], s[2 * kb][1]);
                pw[4 * kb + 1] = pack16<F16>(s[2 * kb][2], s[2 * kb][3]);
                pw[4 * kb + 2] = pack16<F16>(s[2 * kb + 1][0], s[2 * kb + 1][1]);
                pw[4 * kb + 3] = pack16<F16>(s[2 * kb + 1][2], s[2 * kb + 1][3]);
              } else {
                const int t0 = tb + kb * 16 + 2 * c4;
                const int tl = kb * 16 + 2 * c4;
                const float v0 = t0 < valid ? vsc[tl] : 0.f;
                const float v1 = t0 + 1 < valid ? vsc[tl + 1] : 0.f;
                const float v2 = t0 + 8 < valid ? vsc[tl + 8] : 0.f;
                const float v3 = t0 + 9 < valid ? vsc[tl + 9] : 0.f;
                pw[4 * kb] = pack_f16x2(s[2 * kb][0] * v0, s[2 * kb][1] * v1);
                pw[4 * kb + 1] = pack_f16x2(s[2 * kb][2] * v0, s[2 * kb][3] * v1);
                pw[4 * kb + 2] = pack_f16x2(s[2 * kb + 1][0] * v2, s[2 * kb + 1][1] * v3);
                pw[4 * kb + 3] = pack_f16x2(s[2 * kb + 1][2] * v2, s[2 * kb + 1][3] * v3);
              }
            }
          }
          send(pw, al0, al1, 0.f, 0.f);
        }
        stage += it.nst;
        if (FP8) fence_proxy_async_smem();  // the Q slot was rewritten through the generic proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qempty + 8 * qs);
        ++qn;
      }
      // Closing message: the rows' running max and (this lane's) sum.
      uint32_t none[NPW];
#pragma unroll
      for (int i = 0; i < NPW; ++i) none[i] = 0u;
      send(none, m0, m1, l0, l1);
    }
    if (FP8) cp_async_wait<0>();  // no scale copy may still be landing when the CTA exits
    return;
  }

  // ============================================================== PV warps
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* redml = reinterpret_cast<float*>(smem + C::OFF_REDML);
  float acc[NT8][4];
  // Takes one message: NPW P words and four floats.
  auto recv = [&](uint32_t* words, float& a, float& b, float& c, float& d) {
    const int ms = nmsg % NMSG;
    if (ok) {
      ok = mbar_wait(bar_pfull + 8 * (cw * NMSG + ms), (nmsg / NMSG) & 1, kWaitLimitNs, s_abort);
      if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
    }
    const uint4* m = msg_base + ms * (C::MSG / 16);
#pragma unroll
    for (int v = 0; v < NPW / 4; ++v) {
      const uint4 x = m[v * 32];
      words[4 * v] = x.x; words[4 * v + 1] = x.y; words[4 * v + 2] = x.z; words[4 * v + 3] = x.w;
    }
    const uint4 x = m[(NPW / 4) * 32];
    a = __uint_as_float(x.x); b = __uint_as_float(x.y); c = __uint_as_float(x.z); d = __uint_as_float(x.w);
    mbar_arrive(bar_pempty + 8 * (cw * NMSG + ms));
    ++nmsg;
  };

  // Balanced schedule: a sequence with no keys has no work item; CTA
  // b % grid writes its rows (out = 0, lse = -inf).
  if (p.num_splits == 0 && !p.tidar) {
    const int ctid = (warp - PAIRS) * 32 + lane;
    for (int b = blockIdx.x; b < p.B; b += p.grid) {
      if (s_ctx[b] != 0) continue;
      const size_t rows = (size_t)p.T * p.Hq;
      uint4* o4 = reinterpret_cast<uint4*>(p.out + (size_t)b * rows * D);
      for (size_t i = ctid; i < rows * D / 8; i += 64 * PAIRS) o4[i] = make_uint4(0, 0, 0, 0);
      if (p.lse)
        for (size_t i = ctid; i < rows; i += 64 * PAIRS) p.lse[(size_t)b * rows + i] = NEG_INF;
    }
  }

  while (next_item(p, s_ctx, s_start, cur, it)) {
#pragma unroll
    for (int i = 0; i < NT8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    for (int j = 0; j < it.nst; ++j) {
      const int st = stage + j;
      const int slot = st % NS;
      if (ok) {
        ok = mbar_wait(bar_full + 8 * slot, (st / NS) & 1, kWaitLimitNs, s_abort);
        if (!ok && lane == 0) raise_abort(s_abort, p.err_flags);
      }
      if (handled(j)) {
        uint32_t pw[NPW];
        float al0, al1, u0, u1;
        recv(pw, al0, al1, u0, u1);
        if (ok) {
          const bool scr = it.scratch && j == it.nst - 1;
          const int valid = stage_valid(j);
          const int lbt = scr ? 6 : p.lbr;
          const int brows = scr ? p.TP : p.BR;
          const uint32_t box_bytes = (uint32_t)(NCH * H2 * brows * 128);
          const uint32_t cstride = (uint32_t)(H2 * brows * 128);
          const uint32_t hoff = (uint32_t)(hl * brows * 128);
          auto row_base = [&](int tok) -> uint32_t {
            return (uint32_t)(tok >> lbt) * box_bytes + (uint32_t)(tok & ((1 << lbt) - 1)) * 128u + hoff;
          };
          const uint32_t vb_ = sbase + slot * C::STAGE + C::TILE;
          const int sw = lane & 7;
          if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < NT8; ++i) {
              acc[i][0] *= al0;
              acc[i][1] *= al0;
              acc[i][2] *= al1;
              acc[i][3] *= al1;
            }
          }
          // ---- O += P V
          const bool partial = valid < tb + TSL;
#pragma unroll
          for (int kb = 0; kb < NTS / 2; ++kb) {
            const int t0 = tb + kb * 16 + 2 * c4;
            uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
            if (partial) {
              vm0 = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
              vm1 = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
            }
            const uint32_t vrow = vb_ + row_base(tb + kb * 16 + ((lane >> 3) & 1) * 8 + sw);
            const uint32_t* pa = pw + 4 * kb;
            if (!FP8) {
#pragma unroll
              for (int nd = 0; nd < DH / 16; ++nd) {
                const int ndg = hh * (DH / 16) + nd;  // 16-column group of the row
                const int unit = ((ndg * 16) % 64) / 8 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vrow + (ndg / 4) * cstride + ((unit ^ sw) << 4), b0, b1, b2, b3);
                if (partial) {
                  b0 &= vm0; b1 &= vm1; b2 &= vm0; b3 &= vm1;
                }
                mma16<F16>(acc[2 * nd], pa, b0, b1);
                mma16<F16>(acc[2 * nd + 1], pa, b2, b3);
              }
            } else {
#pragma unroll
              for (int uu = 0; uu < DH / 32; ++uu) {
                const int unit = 2 * (hh * (DH / 32) + uu) + (lane >> 4);
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
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    }
    stage += it.nst;
    float m0, m1, l0, l1;
    {
      uint32_t none[NPW];
      recv(none, m0, m1, l0, l1);
    }

    // ---- merge the NGW pairs of each row tile, then write (as in the
    // single-role kernel, among the PV warps)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
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
    auto merge_columns = [&](int i0, int i1) {
#pragma unroll
      for (int i = i0; i < i1; ++i) {
        float a0 = acc[i][0] * w00, a1 = acc[i][1] * w00, a2 = acc[i][2] * w01, a3 = acc[i][3] * w01;
#pragma unroll
        for (int q = 0; q < NGW - 1; ++q) {
          const float* rb = red + (size_t)(hh * (NGW - 1) + q) * C::ROWS * C::RSTR + (i - i0) * 8 + 2 * c4;
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
      for (int ck = 0; ck < DH / C::CHW; ++ck) {
        constexpr int NCT = C::CHW / 8;
        named_barrier_sync(2, 64 * PAIRS);
        if (gi > 0) {
          float* rb = red + (size_t)(hh * (NGW - 1) + gi - 1) * C::ROWS * C::RSTR;
#pragma unroll
          for (int i = 0; i < NCT; ++i) {
            const int ia = ck * NCT + i;
            *reinterpret_cast<float2*>(rb + rho0 * C::RSTR + i * 8 + 2 * c4) = make_float2(acc[ia][0], acc[ia][1]);
            *reinterpret_cast<float2*>(rb + rho1 * C::RSTR + i * 8 + 2 * c4) = make_float2(acc[ia][2], acc[ia][3]);
          }
          if (ck == 0 && c4 == 0 && hh == 0) {
            float* ml = redml + (size_t)(gi - 1) * C::ROWS * 2;
            ml[2 * rho0] = m0;
            ml[2 * rho0 + 1] = l0;
            ml[2 * rho1] = m1;
            ml[2 * rho1 + 1] = l1;
          }
        }
        named_barrier_sync(2, 64 * PAIRS);
        if (gi == 0) {
          if (ck == 0) merge_weights();
          merge_columns(ck * NCT, (ck + 1) * NCT);
        }
      }
    } else {
      merge_weights();
      merge_columns(0, NT8);
    }
    if (gi != 0) continue;
    float lse0 = L0 > 0.f ? (M0 + lg2(L0)) * kLn2 : NEG_INF;
    float lse1 = L1 > 0.f ? (M1 + lg2(L1)) * kLn2 : NEG_INF;
    // An item cut short by a timed-out wait (in any role of the CTA) is
    // written as NaN, so that no part of it passes as a result.
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
      const int rhl = rho / GT, rem = rho - rhl * GT;
      const int t = rem / p.G;
      const int h = (it.hg * H2 + rhl) * p.G + (rem - t * p.G);
      const size_t row = ((size_t)it.b * p.T + t) * p.Hq + h;
      const float lsev = h2 ? lse1 : lse0;
      if (it.part < 0) {
        __nv_bfloat16* o = p.out + row * D + hh * DH;
        if (!FP8) {
#pragma unroll
          for (int i = 0; i < NT8; ++i)
            *reinterpret_cast<uint32_t*>(o + i * 8 + 2 * c4) = pack16<F16>(acc[i][2 * h2], acc[i][2 * h2 + 1]);
        } else {
#pragma unroll
          for (int u = 0; u < DH / 16; ++u)
            *reinterpret_cast<uint2*>(o + 16 * u + 4 * c4) =
                make_uint2(pack_bf16x2(acc[2 * u][2 * h2], acc[2 * u + 1][2 * h2]),
                           pack_bf16x2(acc[2 * u][2 * h2 + 1], acc[2 * u + 1][2 * h2 + 1]));
        }
        if (c4 == 0 && hh == 0 && p.lse) p.lse[row] = lsev;
      } else {
        const size_t prow = p.num_splits > 0 ? row * p.num_splits + it.part : (size_t)it.part * p.M + rho;
        float* o = p.part_o + prow * D + hh * DH;
        if (!FP8) {
#pragma unroll
          for (int i = 0; i < NT8; ++i)
            *reinterpret_cast<float2*>(o + i * 8 + 2 * c4) = make_float2(acc[i][2 * h2], acc[i][2 * h2 + 1]);
        } else {
#pragma unroll
          for (int u = 0; u < DH / 16; ++u)
            *reinterpret_cast<float4*>(o + 16 * u + 4 * c4) =
                make_float4(acc[2 * u][2 * h2], acc[2 * u + 1][2 * h2], acc[2 * u][2 * h2 + 1],
                            acc[2 * u + 1][2 * h2 + 1]);
        }
        if (c4 == 0 && hh == 0) p.part_lse[prow] = lsev;
      }
    }
  }
  launch_dependents();
}

}  // namespace pa
