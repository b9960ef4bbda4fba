// Fifth-generation tensor-core building blocks for sm_103a: shared-memory
// matrix descriptors, the kind::f16 instruction descriptor, tensor-memory
// (TMEM) allocation, single-thread tcgen05.mma issue with completion tracked
// by an mbarrier (bounded wait), tcgen05.ld read-back, and TMA tile loads.
//
// Operand layouts used here are the 128-byte-swizzle canonical layouts:
//   K-major (rows = M or N, 64 bf16 of K per 128-byte row):
//     an atom is 8 rows x 128 B (1024 B, 1024-aligned); the 16-byte chunk c of
//     row r sits at chunk position c ^ (r % 8); atoms of consecutive 8-row
//     groups are SBO bytes apart.  A K-step of 16 elements advances the start
//     address by 32 B inside the atom (the hardware applies the swizzle).
//   MN-major (rows = K, 64 bf16 of M/N per 128-byte row):
//     the same 8 x 128 B atoms, with K rows inside; atoms of consecutive
//     8-row groups along K are SBO bytes apart and atoms along M/N are LBO
//     bytes apart.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace lcsw {

// ------------------------------------------------------------ descriptors ---
// Shared-memory matrix descriptor (64 bit): start address >> 4 in bits 0-13,
// leading byte offset >> 4 in bits 16-29, stride byte offset >> 4 in bits
// 32-45, descriptor version 1 in bits 46-47, base offset 0 (atoms 1024-aligned)
// in bits 49-51, layout type in bits 61-63 (2 = 128-byte swizzle).
constexpr uint32_t kLayoutSwizzle128 = 2;

__host__ __device__ constexpr uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                                 uint32_t layout = kLayoutSwizzle128) {
    return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
           (uint64_t(layout & 7u) << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B and an
// fp32 accumulator: D format (1 = f32) in bits 4-5, A format (1 = bf16) in bits
// 7-9, B format (1 = bf16) in bits 10-12, A / B major-ness (0 = K-major, 1 =
// MN-major) in bits 15 / 16, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) |
           (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Byte offset of element (row, k) of a K-major 128B-swizzled bf16 tile whose
// 8-row atoms are `sbo` bytes apart (k < 64: one atom column).
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t row, uint32_t k, uint32_t sbo) {
    return (row / 8) * sbo + (row % 8) * 128 + ((((k / 8) ^ (row % 8)) & 7u) * 16) + (k % 8) * 2;
}

// ------------------------------------------------------------- mbarrier -----
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// Wait for the phase with the given parity to complete.  Each try suspends
// the thread until the phase completes or kSuspendNs pass (so waiting warps
// do not spin on issue slots); gives up once `budget_ns` nanoseconds of the
// global timer have passed since the first try and returns false.  The bound
// is elapsed time, not a count of tries: a try may return at once.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0u;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          unsigned long long budget_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try(a, parity)) return true;
        if (globaltimer_ns() - t0 > budget_ns) return false;
    }
}

// Arrive once on the mbarrier and expect `bytes` of asynchronous copies.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// -------------------------------------------------------------------- TMA -----
// Tiled 3-D tensor load into shared memory; completion is counted in bytes on
// the mbarrier.  `tmap` is the address of a CUtensorMap kernel parameter.  The
// innermost coordinate must address a 16-byte boundary (here always 0).
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, uint64_t *bar, int c0,
                                            int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Untiled bulk copy of `bytes` contiguous bytes into shared memory (TMA
// engine); completion is counted in bytes on the mbarrier.  Both addresses
// 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------------ TMEM -----
// Allocation and release are warp-wide; the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make generic-proxy writes to shared memory visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One lane of a converged warp (elect.sync): the lane that issues tensor-core
// work, with the descriptors computed warp-uniformly by all lanes.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n .reg .pred p;\n .reg .b32 lane;\n elect.sync lane|p, 0xffffffff;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

// ------------------------------------------------------------------- MMA -----
// D[tmem] (+)= A[smem] * B[smem]; one thread issues.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}
// Arrive once on the mbarrier when every MMA this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------ read-back -----
// Warp w reads TMEM lanes 32*(w%4) .. +31; thread t gets lane 32*(w%4)+t,
// columns col .. col+15 (fp32 bits).  Follow with tc_wait_ld().
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// As tc_ld16, columns col .. col+31.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }


}  // namespace lcsw
