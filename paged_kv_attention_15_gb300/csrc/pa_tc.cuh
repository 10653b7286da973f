// Inline-PTX building blocks for the fifth-generation tensor cores of
// sm_103a (tcgen05): tensor-memory allocation, shared-memory matrix
// descriptors, the kind::f16 MMA with an fp32 accumulator in tensor memory,
// commits to mbarriers, and tensor-memory loads and stores.
#pragma once

#include <cstdint>

namespace pa {

// ------------------------------------------------------- tensor memory
// Allocates `ncols` columns (a power of two >= 32) of this CTA's tensor
// memory; the whole warp executes it and the base address lands in shared
// memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Orders tensor-core operations around a thread synchronisation (an mbarrier
// wait, a CTA or named barrier).
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// --------------------------------------------------------- descriptors
// Shared-memory matrix descriptor: start address, leading- and
// stride-dimension byte offsets (16-byte units), the fixed version field,
// and the swizzle mode (0 none, 2 128-byte, 4 64-byte, 6 32-byte).
// K-major swizzled layouts: rows of one swizzle width, 8-row groups `sbo`
// apart (`lbo` unused). MN-major swizzled layouts: `lbo` between swizzle
// atoms along M/N, `sbo` between 8-row groups along K.
constexpr uint32_t kSwz128 = 2, kSwz64 = 4, kSwz32 = 6;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)(swz & 7u) << 61);
}

// Instruction descriptor of kind::f16 with an fp32 accumulator: M x N, A and
// B both f16 (bf16 = false) or both bf16, each K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn, bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ MMA
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread; `accumulate` = 0
// overwrites D.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier when every MMA this thread issued before has
// completed (their shared-memory reads and tensor-memory writes).
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// ------------------------------------------------- tensor-memory access
// 32x32b shape: thread i of the warp reads lane (quadrant base + i), 16
// consecutive 32-bit columns from `taddr`'s column. The wait for the load
// sits in the same asm statement, so the registers are valid when it ends.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// NC (a multiple of 16) consecutive columns; stores complete at
// tmem_wait_st().
template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
#pragma unroll
  for (int i = 0; i < NC / 16; ++i) tmem_ld16(taddr + 16 * i, v + 16 * i);
}

template <int NC>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float* v) {
#pragma unroll
  for (int i = 0; i < NC / 16; ++i) tmem_st16(taddr + 16 * i, v + 16 * i);
}

// --------------------------------------------------------------- barriers
// CTA-level barrier over `threads` threads that also ORs a predicate across
// them (every participant gets the same result).
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

}  // namespace pa
