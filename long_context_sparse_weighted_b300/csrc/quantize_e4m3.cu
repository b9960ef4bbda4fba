// FP8 (E4M3) pooled indexer keys: bf16 pooled keys -> the tile-major FP8
// cache the FP8 decode step streams (tiles of 16 groups: 16 rows of 64 codes,
// then the 16 rows' fp32 scales; 1088 bytes, 68 per group against 128 in
// bf16).  Arithmetic in e4m3_core.cuh: one scale per 64-value row (amax /
// 448), codes rounded exactly to nearest, ties to the even code.
#include "common.cuh"
#include "e4m3_core.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

// Eight lanes per row, eight values per lane: the row's largest magnitude by
// a shuffle over the eight lanes, then eight codes per lane.
__global__ void __launch_bounds__(256) quantize_keys_kernel(const uint16_t *__restrict__ kp,
                                                            int64_t sp_b, int n_groups,
                                                            uint8_t *__restrict__ kq, int64_t sq_b,
                                                            int64_t rows) {
    const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 8;
    const int sub = threadIdx.x & 7;
    if (row >= rows) return;  // the 8 lanes of a row leave together
    const int b = int(row / n_groups), g = int(row % n_groups);
    const uint4 w = ld_nc16(kp + int64_t(b) * sp_b + int64_t(g) * 64 + sub * 8);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf_lo(ws[i]);
        x[2 * i + 1] = bf_hi(ws[i]);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const unsigned grp = 0xFFu << (threadIdx.x & 24);  // the row's 8 lanes
    amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 4));
    const float sc = e4m3_row_scale(amax);
    uint32_t c[2] = {0u, 0u};
    if (sc != 0.f) {
        const float inv = __frcp_rn(sc);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i / 4] |= e4m3_quantize(x[i], sc, inv) << (8 * (i % 4));
    }
    uint8_t *tile = kq + int64_t(b) * sq_b + int64_t(g / 16) * kE4m3TileBytes;
    *reinterpret_cast<uint2 *>(tile + (g % 16) * 64 + sub * 8) = make_uint2(c[0], c[1]);
    if (sub == 0) *reinterpret_cast<float *>(tile + 1024 + (g % 16) * 4) = sc;
}

}  // namespace

cudaError_t launch_quantize_keys_e4m3(const uint16_t *k_pooled, int64_t sp_b, int B, int n_groups,
                                      uint8_t *kq, int64_t sq_b, cudaStream_t st) {
    const int64_t rows = int64_t(B) * n_groups;
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows * 8 + 255) / 256;
    quantize_keys_kernel<<<unsigned(blocks), 256, 0, st>>>(k_pooled, sp_b, n_groups, kq, sq_b,
                                                           rows);
    return cudaGetLastError();
}

}  // namespace lcsw

namespace lcsw {
namespace {

// A K or V cache row of `width` bf16 values -> width E4M3 codes and the row's
// fp32 scale (the same arithmetic as the pooled keys).  One warp per row: each
// lane takes pairs lane, lane + 32, ... of the row.
__global__ void __launch_bounds__(256) quantize_rows_kernel(
    const uint16_t *__restrict__ x, int64_t sx_b, const int32_t *__restrict__ row_begin,
    int n_rows, int width, int B, uint8_t *__restrict__ codes, int64_t sc_b,
    float *__restrict__ scales, int64_t ss_b) {
    const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= int64_t(B) * n_rows) return;  // the whole warp leaves together
    const int b = int(wid / n_rows);
    const int64_t r = (row_begin ? int64_t(__ldg(row_begin + b)) : 0) + wid % n_rows;
    if (r < 0) return;
    const uint16_t *xr = x + int64_t(b) * sx_b + r * width;
    const int npair = width / 2;
    float amax = 0.f;
    for (int p = lane; p < npair; p += 32) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(xr) + p);
        amax = fmaxf(amax, fmaxf(fabsf(bf_lo(w)), fabsf(bf_hi(w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = e4m3_row_scale(amax);
    const float inv = sc != 0.f ? __frcp_rn(sc) : 0.f;
    uint8_t *cr = codes + int64_t(b) * sc_b + r * width;
    for (int p = lane; p < npair; p += 32) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(xr) + p);
        uint32_t c = 0u;
        if (sc != 0.f) c = e4m3_quantize(bf_lo(w), sc, inv) | (e4m3_quantize(bf_hi(w), sc, inv) << 8);
        *reinterpret_cast<uint16_t *>(cr + 2 * p) = uint16_t(c);
    }
    if (lane == 0) scales[int64_t(b) * ss_b + r] = sc;
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const uint16_t *x, int64_t sx_b, const int32_t *row_begin,
                                      int n_rows, int width, int B, uint8_t *codes, int64_t sc_b,
                                      float *scales, int64_t ss_b, cudaStream_t st) {
    const int64_t warps = int64_t(B) * n_rows;
    if (warps == 0) return cudaSuccess;
    quantize_rows_kernel<<<unsigned((warps * 32 + 255) / 256), 256, 0, st>>>(
        x, sx_b, row_begin, n_rows, width, B, codes, sc_b, scales, ss_b);
    return cudaGetLastError();
}

}  // namespace lcsw
