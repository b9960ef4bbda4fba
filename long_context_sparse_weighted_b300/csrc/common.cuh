// Device helpers shared by the liblcsw kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lcsw {

constexpr int kWarp = 32;

// ------------------------------------------------------------------ bf16 ---

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    return uint32_t(f2bf(lo)) | (uint32_t(f2bf(hi)) << 16);
}

// ---------------------------------------------------------- memory access ---

// 16-byte load that bypasses L1 allocation (streamed data, read once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_nc16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async 16 bytes global -> shared; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
// cp.async 4 bytes global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// ------------------------------------------------------------ tensor core ---

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// ------------------------------------------------------------ selection ----

// Order-preserving map fp32 -> uint32: a > b (as reals) iff key(a) > key(b);
// -0 and +0 map to the same key.  NaN is not supported.
__device__ __forceinline__ uint32_t score_key(float s) {
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ----------------------------------------------------------- block scans ---

// Exclusive prefix sum over the block (blockDim.x a multiple of 32, <= 1024).
// `scratch` holds at least 33 ints.  Returns the exclusive prefix of `v`; the
// block total is written to *total.  Contains __syncthreads().
__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nwarps) scratch[lane] = w;  // inclusive warp totals
        if (lane == nwarps - 1) scratch[32] = w;
    }
    __syncthreads();
    int before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
    *total = scratch[32];
    __syncthreads();
    return before;
}

// ---------------------------------------------------------- bounds checks ---
// Built with -DLCSW_CHECKS=1, the kernels check their data-dependent indices
// (positions derived from candidate counts, selections and lengths) against
// the extents they were given: a failed check records its code in this
// translation unit's check word (the first failure wins) and the access is
// skipped -- no trap.  lcsw_check_status() collects and clears the words.  In
// the normal build LCSW_INBOUNDS(cond, code) is the constant true.
void register_check_reader(int (*reader)());  // lcsw_api.cu
#ifdef LCSW_CHECKS
namespace {
__device__ int g_lcsw_check_word;
int lcsw_read_check_word() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_lcsw_check_word, sizeof v) != cudaSuccess) return -1;
    if (v) {
        const int z = 0;
        cudaMemcpyToSymbol(g_lcsw_check_word, &z, sizeof z);
    }
    return v;
}
struct CheckReaderRegistration {
    CheckReaderRegistration() { register_check_reader(&lcsw_read_check_word); }
};
const CheckReaderRegistration g_lcsw_check_registration;
__device__ __forceinline__ bool lcsw_inbounds(bool ok, int code) {
    if (!ok) atomicCAS(&g_lcsw_check_word, 0, code);
    return ok;
}
}  // namespace
#define LCSW_INBOUNDS(cond, code) lcsw_inbounds((cond), (code))
#else
#define LCSW_INBOUNDS(cond, code) true
#endif

// ------------------------------------------------------ bounded waiting ----

// Budget for device-side spin waits, in SM clock cycles (~0.5 s at 2 GHz).
constexpr long long kSpinBudget = 1000000000LL;

// Nanoseconds of the GPU-wide global timer (comparable across SMs).
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Budget for a wait on an mbarrier (tensor-core completion, bulk copies), in
// nanoseconds of the global timer: about one second.
constexpr unsigned long long kWaitNs = 1000000000ull;

}  // namespace lcsw
