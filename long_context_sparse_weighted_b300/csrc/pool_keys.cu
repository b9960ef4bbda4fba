// IndexPool: merge each group of P consecutive cached indexer keys into one
// pooled key by weighted pooling (reading notes "GLM-5.3-Flash: Hybrid
// Attention, IndexPool, and Vision-in-the-Loop", section 2, sub-head
// "IndexPool"; index_kpool 4 in "G2C Brief -- GLM-5.3-Flash", DSA section).
//
//   kbar[b][g][i] = bf16( sum_{j<P} alpha[b][g][j] * k[b][P*g+j][i] )
//
// The result is the exact sum rounded once to bf16, nearest with ties to even:
// an fp32 fma chain with an error bound decides the rounding when no bf16
// boundary lies within the bound, and error-free product and sum
// transformations decide the rest (pool_core.cuh).
//
// Memory: a pure stream.  One thread owns 16 bytes (8 dims) of one group's
// output row and issues P independent 16-byte coalesced loads (one per source
// row; the 8 threads of a row read 128 contiguous bytes), so the bound is HBM
// bandwidth: P*d*2 + P*4 bytes read and d*2 bytes written per group.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "pool_core.cuh"

namespace lcsw {
namespace {

template <int P>
__global__ void __launch_bounds__(256) pool_keys_kernel(
    const uint16_t *__restrict__ k_idx, int64_t sk_b, const float *__restrict__ pool_w,
    int64_t sw_b, const int32_t *__restrict__ seq_len, const int32_t *__restrict__ g_begin,
    int B, int g_span, int d_idx, int cpr_shift, int mode, int tail,
    uint16_t *__restrict__ k_pooled, int64_t sp_b) {
    const int cpr = d_idx >> 3;  // 16-byte chunks per key row
    const int64_t per_b = int64_t(g_span) * cpr;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    // blockIdx.y walks the sequences, blockIdx.x the chunks of one sequence
    for (int b = blockIdx.y; b < B; b += gridDim.y) {
        const int L = __ldg(seq_len + b);
        const int64_t G = L / P;
        int64_t g0;
        if (mode == 1)
            g0 = (L % P == 0 && G > 0) ? G - 1 : G;
        else if (mode == 2)
            g0 = (L > tail ? L - tail : 0) / P;
        else
            g0 = g_begin ? int64_t(__ldg(g_begin + b)) : 0;
        const int64_t n = min(per_b, (G - g0) * cpr);  // chunks that exist
        const uint16_t *src_b = k_idx + int64_t(b) * sk_b;
        const float *w_b = pool_w + int64_t(b) * sw_b;
        uint16_t *dst_b = k_pooled + int64_t(b) * sp_b;
        for (int64_t it = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; it < n; it += stride) {
            int64_t gi;
            int c;
            if (cpr_shift >= 0) {
                gi = it >> cpr_shift;
                c = int(it & (cpr - 1));
            } else {
                gi = it / cpr;
                c = int(it - gi * cpr);
            }
            const int64_t g = g0 + gi;
            if (g < 0) continue;  // a negative g_begin: only existing groups are written
            const uint16_t *src = src_b + (g * P) * d_idx + c * 8;
            uint4 rows[P];
#pragma unroll
            for (int j = 0; j < P; ++j) rows[j] = ld_stream16(src + int64_t(j) * d_idx);
            float a[P];
#pragma unroll
            for (int j = 0; j < P; ++j) a[j] = __ldg(w_b + g * P + j);
            const uint4 o = pool_chunk_fast<P>(a, rows);
            // (with one sequence the strides bound nothing)
            if (LCSW_INBOUNDS(B == 1 || (g + 1) * d_idx <= sp_b, 301))
                *reinterpret_cast<uint4 *>(dst_b + g * d_idx + c * 8) = o;
        }
    }
}

}  // namespace

cudaError_t launch_pool_keys(const uint16_t *k_idx, int64_t sk_b, const float *pool_w,
                             int64_t sw_b, const int32_t *seq_len, const int32_t *g_begin,
                             int B, int g_span, int d_idx, int P, int mode, int tail,
                             uint16_t *k_pooled, int64_t sp_b, cudaStream_t st) {
    const int cpr = d_idx / 8;
    const int64_t per_b = int64_t(g_span) * cpr;
    if (per_b == 0 || B == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 256;
    const int by = B < 65535 ? B : 65535;
    const int cpr_shift = (cpr & (cpr - 1)) == 0 ? __builtin_ctz(unsigned(cpr)) : -1;
    // one wave: the resident blocks of every SM over the whole grid
    static int occ_cache[9];  // per P (a benign race: every thread computes the same value)
    auto grid_x = [&](const void *kern) {
        int occ = occ_cache[P];
        if (occ < 1) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, 0) !=
                    cudaSuccess ||
                occ < 1)
                occ = 4;
            occ_cache[P] = occ;
        }
        const int64_t cap = std::max<int64_t>(1, int64_t(sms) * occ / by);
        return unsigned(std::min<int64_t>((per_b + threads - 1) / threads, cap));
    };
#define LCSW_POOL(PP)                                                                         \
    {                                                                                         \
        auto kern = pool_keys_kernel<PP>;                                                     \
        kern<<<dim3(grid_x(reinterpret_cast<const void *>(kern)), unsigned(by)), threads, 0,  \
               st>>>(k_idx, sk_b, pool_w, sw_b, seq_len, g_begin, B, g_span, d_idx, cpr_shift, \
                     mode, tail, k_pooled, sp_b);                                             \
    }
    switch (P) {
        case 1: LCSW_POOL(1); break;
        case 2: LCSW_POOL(2); break;
        case 4: LCSW_POOL(4); break;
        case 8: LCSW_POOL(8); break;
        default: return cudaErrorInvalidValue;
    }
#undef LCSW_POOL
    return cudaGetLastError();
}

}  // namespace lcsw
