// kvc_tcgen05.cuh -- inline-PTX wrappers for the fifth-generation tensor cores
// of sm_100-class GPUs (tcgen05): tensor-memory (TMEM) allocation, the
// shared-memory matrix descriptors and instruction descriptor of an MMA, the
// MMA itself, its completion (commit to an mbarrier), and the TMEM <->
// register moves of the epilogue.  One instruction per wrapper, written from
// the PTX ISA; the layouts they assume are stated beside each.
#pragma once

#include <cstdint>

namespace kvc {
namespace tc {

// ---- tensor memory -------------------------------------------------------
// Allocate `ncols` TMEM columns (a power of two >= 32) for this CTA; the
// base address is written to shared memory at `dst`.  Executed by one whole
// warp, which must later free them with dealloc.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}

// Let other CTAs on this SM allocate once this CTA's allocation is done.
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations around a thread synchronisation (barrier or
// mbarrier): `before` ahead of the arrive, `after` behind the wait.
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- descriptors -----------------------------------------------------------
// Shared-memory matrix descriptor with the 128-byte swizzle.  The operand is
// stored in swizzle atoms of 8 rows x 128 bytes (1024 bytes, 1024-byte
// aligned); within a row the 16-byte chunk c sits at chunk c ^ (row mod 8),
// which is what a TMA box with CU_TENSOR_MAP_SWIZZLE_128B writes.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  0b001 (descriptor version of sm_100)
//   bits 49-51  base offset (0: atoms 1024-byte aligned)
//   bits 61-63  layout: 2 = 128-byte swizzle
// K-major operand (rows along M or N, the contraction dimension contiguous):
//   sbo = bytes between consecutive 8-row groups (1024 when rows are packed),
//   lbo unused; an MMA step of 16 elements advances the start by 32 bytes
//   inside the 128-byte row.
// MN-major operand (M or N contiguous in 64-element, 128-byte runs; rows
// along the contraction dimension): lbo = bytes between consecutive
// 64-element runs along M/N, sbo = bytes between consecutive 8-row groups
// along the contraction dimension.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of tcgen05.mma .kind::f16 with fp32 accumulation:
//   bits 4-5   D format (1: f32)
//   bits 7-9   A format, bits 10-12 B format (0: f16, 1: bf16)
//   bit 15     A major (0: K-major, 1: MN-major); bit 16 the same for B
//   bits 17-22 N >> 3; bits 24-28 M >> 4
// A and B always have the same 16-bit type here.
__host__ __device__ constexpr uint32_t idesc_f16_f32acc(bool bf16, int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (uint32_t(bf16) << 7) | (uint32_t(bf16) << 10) | (uint32_t(a_mn_major) << 15) |
           (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// ---- the MMA ---------------------------------------------------------------
// D[tmem] = A * B (+ D when `accumulate`), A and B in shared memory by
// descriptor; issued by one thread, asynchronous.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] = A * B (+ D when `accumulate`) with A in tensor memory (row m of
// A in lane m, consecutive K elements along the columns, two 16-bit elements
// per 32-bit column, the lower-indexed one in the low half) and B in shared
// memory by descriptor; issued by one thread, asynchronous.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on the mbarrier when every tcgen05.mma this thread issued so
// far has completed.
__device__ __forceinline__ void commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

// ---- TMEM <-> registers ----------------------------------------------------
// 32 lanes x 32 columns of 32-bit values: thread i of the warp moves lane
// (lane field of taddr) + i, columns [col, col + 32).  A warp may only touch
// the lane quarter 32 * (warp id mod 4).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Wait until this thread's earlier tcgen05.ld (st) have completed.
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Make the compiler treat 32 registers as redefined here, so that no use of
// a tcgen05.ld result is scheduled ahead of the wait that precedes this.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

}  // namespace tc
}  // namespace kvc
