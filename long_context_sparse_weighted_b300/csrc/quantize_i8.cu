// INT8 K/V cache rows: a bf16 K or V cache row of `width` values -> width
// int8 codes and the row's fp32 scale (arithmetic in i8_core.cuh).  One warp
// per row: the row's largest magnitude by shuffles, then each lane codes the
// pairs lane, lane + 32, ... of the row.
#include "common.cuh"
#include "i8_core.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

__global__ void __launch_bounds__(256) quantize_rows_i8_kernel(
    const uint16_t *__restrict__ x, int64_t sx_b, const int32_t *__restrict__ row_begin,
    int n_rows, int width, int B, int8_t *__restrict__ codes, int64_t sc_b,
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
    const float sc = i8_row_scale(amax);
    const float inv = sc != 0.f ? __frcp_rn(sc) : 0.f;
    int8_t *cr = codes + int64_t(b) * sc_b + r * width;
    for (int p = lane; p < npair; p += 32) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(xr) + p);
        uint32_t c = 0u;
        if (sc != 0.f)
            c = (uint32_t(i8_quantize(bf_lo(w), sc, inv)) & 0xFFu) |
                ((uint32_t(i8_quantize(bf_hi(w), sc, inv)) & 0xFFu) << 8);
        *reinterpret_cast<uint16_t *>(cr + 2 * p) = uint16_t(c);
    }
    if (lane == 0) scales[int64_t(b) * ss_b + r] = sc;
}

}  // namespace

cudaError_t launch_quantize_rows_i8(const uint16_t *x, int64_t sx_b, const int32_t *row_begin,
                                    int n_rows, int width, int B, int8_t *codes, int64_t sc_b,
                                    float *scales, int64_t ss_b, cudaStream_t st) {
    const int64_t warps = int64_t(B) * n_rows;
    if (warps == 0) return cudaSuccess;
    quantize_rows_i8_kernel<<<unsigned((warps * 32 + 255) / 256), 256, 0, st>>>(
        x, sx_b, row_begin, n_rows, width, B, codes, sc_b, scales, ss_b);
    return cudaGetLastError();
}

}  // namespace lcsw
