/*
 * pa_decode.h - C ABI of the GB300 (sm_103a) paged-KV decode attention engine.
 *
 * The operation: softmax attention of a few query tokens per sequence over a
 * KV cache stored in fixed-size physical pages and addressed through a
 * per-sequence block table, with grouped query heads, split-K partials
 * combined by their log-sum-exp, an fp8 e4m3fn cache with per-token scales,
 * and a draft-block (TiDAR) mode with extra contiguous scratch KV.
 * Sources: ROCm blog "Implementing a High-Performance Custom Diffusion
 * Attention Kernel with FlyDSL" (introduction, items 1-3: paged KV caches,
 * scratch storage for speculatively generated tokens, FlashAttention and
 * split-K; section Graph Capture: runtime versus fixed parameters) and the
 * MSLK pull request "[ROCm] Add FlyDSL paged-attention decode backend
 * (dense + fp8) with benchmark" (section Kernels: dense decode, native fp8
 * decode with symmetric per-token scale, split-K reduce, stream threaded
 * through compute and reduce launches so the calls can be graph-captured).
 *
 * Definition computed, for every sequence b < B, query token t < T and query
 * head h < Hq, with kv head g = h / G and G = Hq / Hkv:
 *   keys j < C_b = context_lens[b]; key j lives in physical page
 *   block_tables[b][j / P], slot j % P, kv head g;
 *   s_j = scale * <q[b][t][h], k_j>;  out = sum_j softmax(s)_j v_j;
 *   lse = ln sum_j exp(s_j)   (natural log, scale included).
 * An empty key set gives out = 0 and lse = -inf.
 *
 * Common conventions
 *  - Every pointer argument is a DEVICE pointer on the current CUDA device,
 *    16-byte aligned; every tensor is dense row-major (contiguous).
 *  - Layouts: q, out [B, T, Hq, D] bf16; k_cache, v_cache
 *    [num_pages, P, Hkv, D] (bf16, or e4m3fn bytes); k_scale, v_scale
 *    [num_pages, P, Hkv] fp32; block_tables [B, max_blocks_per_seq] int32;
 *    context_lens [B] int32; lse [B, T, Hq] fp32; k_scratch, v_scratch
 *    [B, T, Hkv, D] bf16.
 *  - context_lens[b] is clamped on the device to [0, max_blocks_per_seq * P];
 *    only the first ceil(C_b / P) block-table entries of a row are read.
 *    A page id outside [0, num_pages) reads zeros (the copy engine fills
 *    out-of-range boxes); it never faults.
 *  - Ownership: the caller owns every buffer, including the workspace. The
 *    library allocates nothing, keeps no pointer after return, performs no
 *    host<->device copy and no synchronisation. Work is enqueued on `stream`
 *    and completes asynchronously. Calls may be captured into a CUDA graph;
 *    the first call on a device does one-time set-up (device attribute
 *    queries, kernel attributes), so make it before capturing.
 *  - Errors: argument and shape problems are reported BEFORE any launch
 *    (out, lse and the workspace are untouched). PA_ERR_CUDA reports a
 *    launch failure (cudaGetLastError). Nothing aborts or throws across the
 *    ABI. A device-side wait that runs out of time (a bug, never expected)
 *    makes the kernel stop early: every query row whose work was cut short
 *    gets NaN in out and lse (also through the split-K combine), so no part
 *    of an aborted call can pass as a result, and a flag is set that
 *    pa_decode_device_error() reads.
 *
 * Supported: D in {64, 128, 256} (fp8: {128, 256}); P in {16, 32, 64, 128,
 * 256}; M = G * T <= 64 query rows per kv head (more than 32 rows: D in {64,
 * 128}, 16-bit pages).
 * Anything else returns PA_ERR_UNSUPPORTED.
 *
 * num_splits:
 *   0   auto. The flattened list of (sequence, kv head, page) work is cut into
 *       equal contiguous shares, one per CTA of a grid that fills the SMs, so
 *       sequences of any length mix are balanced; a dependent launch combines
 *       the sequences split between CTAs. With so many sequences that their
 *       table does not fit in shared memory, it runs the explicit split count
 *       pa_decode_choose_splits() reports instead. Needs the workspace of
 *       pa_decode_workspace_size(shape, 0) (its layout is private).
 *   1   one CTA per (sequence, kv head) writes out/lse directly; no workspace.
 *   S>1 split s of sequence b covers pages [s*pps, min((s+1)*pps, n_b)),
 *       pps = ceil(n_b / S), n_b = ceil(C_b / P); draft-block scratch tokens
 *       belong to split S-1. The workspace holds, at byte 0, part_out
 *       float [B][T][Hq][S][D] (each split normalised over its own keys) and,
 *       at byte align256(B*T*Hq*S*D*4), part_lse float [B][T][Hq][S]
 *       (-inf for an empty split); pa_decode_reduce() then combines them.
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. NULL = legacy stream. */
typedef struct CUstream_st* pa_stream_t;

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad shape, bad scale */
  PA_ERR_UNSUPPORTED = 2, /* valid but outside the compiled kernel set */
  PA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  PA_ERR_CUDA = 4         /* a CUDA runtime call or launch failed */
} pa_status;

typedef struct pa_shape {
  int32_t batch;              /* B >= 0 (0: nothing to do) */
  int32_t q_tokens;           /* T >= 1: 1 for decode, the draft length for TiDAR */
  int32_t num_q_heads;        /* Hq >= 1, a multiple of num_kv_heads */
  int32_t num_kv_heads;       /* Hkv >= 1 */
  int32_t head_dim;           /* D */
  int32_t page_size;          /* P, tokens per physical page */
  int32_t num_pages;          /* physical pages in each cache tensor, >= 1 */
  int32_t max_blocks_per_seq; /* columns of block_tables, >= 1 */
} pa_shape;

/* Bytes of workspace pa_decode* needs for this shape and num_splits (0 for
 * num_splits == 1). For num_splits == 0 the size is the largest over every
 * decode entry point (bf16, f16, fp8, draft block) and every kernel
 * selection (pa_decode_set_kernel_path), and depends on the current
 * device's SM count: size it on the device that will run the call
 * (another GPU model may need more and would return PA_ERR_WORKSPACE).
 * Returns 0 as well for an invalid shape. */
size_t pa_decode_workspace_size(const pa_shape* shape, int32_t num_splits);

/* What num_splits == 0 resolves to on the current device, for this shape and
 * KV format (fp8_kv: 0 for bf16 pages, as pa_decode and pa_decode_tidar;
 * 1 for pa_decode_fp8). Returns 0 when it runs the balanced schedule (one
 * CTA per SM, each taking an equal share of all the shape's pages, so a
 * sequence is split wherever two shares meet), or the explicit split count
 * S >= 1 it falls back to when the per-sequence table does not fit in
 * shared memory (S = ceil(2 * SMs / (B * kv head groups)), at most
 * max_blocks_per_seq). Returns -1 for an invalid or unsupported shape, or
 * when no CUDA device is usable. This is the split scheduler behind
 * num_splits = 0 (the MSLK pull request's review: "num_splits: int = 0"):
 * the grid fills the SMs. */
int32_t pa_decode_choose_splits(const pa_shape* shape, int32_t fp8_kv);

/* Dense bf16 paged decode (the MSLK page's dense decode kernel).
 * q, k_cache, v_cache, out: bf16 as above. lse may be NULL. scale: the
 * softmax scale (finite), e.g. 1/sqrt(D). */
pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens,
                    const pa_shape* shape, float scale, void* out, float* lse,
                    int32_t num_splits, void* workspace, size_t workspace_bytes,
                    pa_stream_t stream);

/* Native fp8 paged decode (the MSLK page's fp8 kernel: OCP e4m3fn codes with
 * a symmetric per-token, per-kv-head fp32 scale; value = code * scale).
 * q is bf16 and is not quantised. The codes are converted exactly in
 * registers; the products run in f16 with fp32 accumulation, so |q| must be
 * below 65504. Otherwise as pa_decode. */
pa_status pa_decode_fp8(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                        const float* k_scale, const float* v_scale,
                        const int32_t* block_tables, const int32_t* context_lens,
                        const pa_shape* shape, float scale, void* out, float* lse,
                        int32_t num_splits, void* workspace, size_t workspace_bytes,
                        pa_stream_t stream);

/* Dense f16 paged decode: as pa_decode with q, k_cache, v_cache and out in
 * IEEE binary16 (the MSLK page's dense path takes f16 or bf16); the products
 * run in f16 with fp32 accumulation. */
pa_status pa_decode_f16(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens,
                        const pa_shape* shape, float scale, void* out, float* lse,
                        int32_t num_splits, void* workspace, size_t workspace_bytes,
                        pa_stream_t stream);

/* Draft-block (TiDAR) decode: as pa_decode, plus the T scratch tokens of each
 * sequence (k_scratch, v_scratch [B, T, Hkv, D] bf16, contiguous) as extra
 * keys after the paged prefix. Every draft token attends to the whole prefix
 * and to all T scratch tokens (no mask inside the draft block); C_b counts
 * the paged prefix only. (ROCm blog, introduction item 1.) */
pa_status pa_decode_tidar(const void* q, const void* k_cache, const void* v_cache,
                          const void* k_scratch, const void* v_scratch,
                          const int32_t* block_tables, const int32_t* context_lens,
                          const pa_shape* shape, float scale, void* out, float* lse,
                          int32_t num_splits, void* workspace, size_t workspace_bytes,
                          pa_stream_t stream);

/* Block-masked draft-block (TiDAR) decode: as pa_decode_tidar, but draft
 * token t sees only the scratch tokens t' with t' / draft_block <=
 * t / draft_block (integer division): the first
 * min(T, (t / draft_block + 1) * draft_block) of them. draft_block = 1 is a
 * causal draft, draft_block >= T the unmasked pa_decode_tidar; draft_block
 * < 1 is PA_ERR_INVALID_ARG. The paged prefix stays visible to every draft
 * token. The ROCm blog leaves the mask inside the draft block open
 * (introduction items 1-2: a highly configurable attention pattern); this is
 * the block-causal family of it. */
pa_status pa_decode_tidar_masked(const void* q, const void* k_cache, const void* v_cache,
                                 const void* k_scratch, const void* v_scratch,
                                 const int32_t* block_tables, const int32_t* context_lens,
                                 const pa_shape* shape, float scale, int32_t draft_block, void* out,
                                 float* lse, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                 pa_stream_t stream);

/* Split-K combine (the MSLK page's pa_decode_reduce): for every (b, t, h),
 * M = max_s lse_s, w_s = exp(lse_s - M), out = sum_s w_s part_out_s / sum_s w_s,
 * lse = M + ln sum_s w_s; all splits empty gives out = 0, lse = -inf.
 * part_out float [B][T][Hq][num_splits][D], part_lse float [B][T][Hq][num_splits]
 * (the layout pa_decode writes for num_splits > 1). out bf16 [B][T][Hq][D];
 * lse may be NULL. num_splits >= 1. Only batch, q_tokens, num_q_heads and
 * head_dim of shape are used (head_dim a multiple of 4, <= 1024). A split
 * whose lse is NaN makes its row NaN. */
pa_status pa_decode_reduce(const float* part_out, const float* part_lse, int32_t num_splits,
                           const pa_shape* shape, void* out, float* lse, pa_stream_t stream);

/* pa_decode_reduce with out in IEEE binary16: the combine for callers of
 * pa_decode_f16 that run explicit splits and combine the partials
 * themselves (the MSLK page's dense path is f16 or bf16). Arguments, layouts
 * and errors as pa_decode_reduce. */
pa_status pa_decode_reduce_f16(const float* part_out, const float* part_lse, int32_t num_splits,
                               const pa_shape* shape, void* out, float* lse, pa_stream_t stream);

/* KV-cache append, the step before a decode: writes the T = shape->q_tokens
 * new tokens of every sequence into its pages (the ROCm blog's paged cache,
 * introduction item 1). Token t of sequence b takes logical position
 * j = C_b + t, C_b = context_lens[b] (the tokens already cached, clamped to
 * [0, max_blocks_per_seq * P]): slot j % P of page block_tables[b][j / P].
 * For every kv head g the row k_new[b][t][g][:] (v_new likewise) goes to
 * k_cache[page][slot][g][:].
 *  - k_new, v_new: bf16 [B, T, Hkv, D], contiguous; k_cache, v_cache: bf16
 *    [num_pages, P, Hkv, D]. D in {64, 128, 256}; num_q_heads is not used.
 *    The rows are copied bit for bit, so f16 rows into f16 caches (the
 *    caches of pa_decode_f16) take the same call.
 *  - context_lens is read, not advanced: the caller adds T after the call.
 *  - Positions at or past max_blocks_per_seq * P, and page ids outside
 *    [0, num_pages), are skipped (nothing written, no fault).
 *  - Rows of two (b, t) that land in the same slot: one of them wins.
 * Errors as for pa_decode; no workspace, no allocation, graph-capturable. */
pa_status pa_kv_append(const void* k_new, const void* v_new, const int32_t* block_tables,
                       const int32_t* context_lens, const pa_shape* shape, void* k_cache, void* v_cache,
                       pa_stream_t stream);

/* fp8 KV-cache append: as pa_kv_append, quantising each written row (token,
 * kv head) to OCP e4m3fn with its own symmetric scale, computed when the
 * cache is written (the MSLK page: native fp8 with a symmetric per-token
 * scale, OCP e4m3fn; its review asks for scales at write time). With x the
 * bf16 row widened to float32:
 *     scale = amax_d |x_d| / 448   (IEEE float32 division; 1 if amax = 0)
 *     code_d = e4m3fn(x_d / scale) (float32 division, round to nearest even,
 *                                   magnitudes past 448 saturate to 448)
 * scale goes to k_scale[page][slot][g] (v_scale likewise), fp32
 * [num_pages, P, Hkv], the layout pa_decode_fp8 reads. x must be finite. */
pa_status pa_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* block_tables,
                           const int32_t* context_lens, const pa_shape* shape, uint8_t* k_cache, uint8_t* v_cache,
                           float* k_scale, float* v_scale, pa_stream_t stream);

/* pa_decode without a caller-provided workspace (the papers have no
 * counterpart; this is a convenience of this library). Some callers cannot
 * allocate device memory at the point where they decode: a plug-in that is
 * handed only the input and output pointers by a host framework whose own
 * memory pool has reserved the device, or a latency-critical path that must
 * not call cudaMalloc because it can block and synchronise the device. This
 * entry point takes the same arguments as pa_decode minus the workspace and
 * keeps the split-K partials in a fixed scratch array that the library
 * reserves statically on every GPU that loads it (held until the process
 * exits): PA_NOALLOC_SCRATCH_BYTES bytes. It allocates nothing.
 *  - The limit applies to the partials pa_decode itself uses for this shape
 *    and num_splits on this device. pa_decode_workspace_size(shape, S) is
 *    that size for S >= 1; for S = 0 it is the largest over every decode
 *    format, so it may exceed what this bf16 call needs. Calls over the
 *    limit return PA_ERR_WORKSPACE before any launch.
 *  - The first call on a device looks up the scratch array's device address
 *    (once per device, with that device current); make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents; nothing in it needs to start at zero (every partial is
 *    written before it is read within a call). Calls whose work overlaps on
 *    the GPU (several streams, or several host threads) race on it: order
 *    them on one stream. */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)
pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            const pa_shape* shape, float scale, void* out, float* lse,
                            int32_t num_splits, pa_stream_t stream);

/* Kernel selection. The decode entry points run one of four split kernels:
 * 1 = warp-level MMA kernel (mma.sync tiles of query rows, every shape the
 *     library supports),
 * 2 = token-major tcgen05 kernel (scores and output transposed in tensor
 *     memory; units of 16 or 32 query rows per kv head, D = 128, and fp8
 *     D = 256),
 * 3 = query-row-major tcgen05 kernel (bf16 and f16 caches, D = 128, units of
 *     64 query rows: G * T = 32 with two kv heads per unit, or G * T = 64;
 *     pages of at least 16 tokens), or
 * 4 = warp-level MMA kernel with paired consumer roles (one warp computes
 *     scores, softmax and the P operand, two more P V and the output; fp8
 *     caches with up to 32 query rows per kv head, and 16-bit caches at
 *     D = 128 with units of 33-64 query rows).
 * pa_decode_set_kernel_path(0) (the default) picks per call the kernel
 * measured fastest for the shape (4 for fp8 caches where it has an
 * instance, else 1: the 16-bit units of kernel 4 measured slower); 1 forces the warp-level kernel; 2, 3 and 4 use that
 * kernel wherever it has an instance (else the warp-level kernel). Process-wide, for tests and benchmarks; the results agree within
 * rounding. Returns PA_ERR_INVALID_ARG for any other value. */
pa_status pa_decode_set_kernel_path(int32_t path);

/* Split-K combine of the balanced schedule (num_splits == 0): mode 0 (the
 * default) runs a separate combine kernel after the split kernel (launched
 * with programmatic dependent launch); mode 1 fuses it into the warp-level
 * split kernel: each CTA counts its finished piece of a (sequence, kv head
 * group) unit in the workspace, and the last one to finish combines the
 * unit's pieces (one memset of the counters per call replaces the combine
 * launch; fp8 caches, the eight-warp draft-block instances and the
 * tcgen05 kernels keep the separate combine).
 * Measured slower than mode 0 on every benchmark workload. Source: the MSLK
 * pull request "[ROCm] Add FlyDSL paged-attention decode backend (dense +
 * fp8) with benchmark" (Kernels: the split-K partial combine). Results
 * agree within rounding. Process-wide; PA_ERR_INVALID_ARG for other values.
 * Host-only. */
pa_status pa_decode_set_combine(int32_t mode);

/* Which kernel (1 to 4, as above) a decode of this shape would run under the
 * current setting; format: 0 bf16 (pa_decode), 1 fp8 (pa_decode_fp8), 2 f16
 * (pa_decode_f16), 3 draft block (pa_decode_tidar*). -1 for an unsupported
 * shape. Host-only. */
int32_t pa_decode_kernel_for(const pa_shape* shape, int32_t format);

/* How many kv heads one work unit of that decode takes (the query rows of
 * those heads share each page's copy: 1, 2, 4 or 8, dividing num_kv_heads),
 * under the current setting; format as for pa_decode_kernel_for. -1 for an
 * unsupported shape. Host-only. */
int32_t pa_decode_heads_per_unit(const pa_shape* shape, int32_t format);

/* A static description of a status code (never NULL). */
const char* pa_status_string(pa_status status);

/* Benchmark hook. Arms the calling thread's NEXT pa_decode, pa_decode_fp8 or
 * pa_decode_tidar call to record `start_event` on its stream just before the
 * split kernel's launch and `split_done_event` just after it (both are
 * cudaEvent_t handles owned by the caller; NULL disarms). The arming is
 * consumed by that call whatever its outcome, so the split kernel alone can
 * be timed with cudaEventElapsedTime. Pure host bookkeeping; no device work. */
pa_status pa_decode_profile_events(void* start_event, void* split_done_event);

/* Reads and clears the current device's error flags set by the kernels
 * (bit 0: a pipeline wait in the split kernel ran out of time). Synchronous;
 * for diagnostics only, never inside stream capture. */
pa_status pa_decode_device_error(int32_t* flags);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
