// INT8 tier of the cache quantization of the serving stack (reading notes
// "GLM-5.3-Flash: Hybrid Attention, IndexPool, and Vision-in-the-Loop",
// section "The serving stack": caches quantized per tier to INT8, FP8 or BF16;
// the pages give no format).  The reading: symmetric codes in [-127, 127],
// one fp32 scale per row = amax / 127, code = the integer nearest to
// x / scale with ties to the even integer.
#pragma once
#include "common.cuh"

namespace lcsw {

// Scale of a row from its largest magnitude: amax / 127 rounded to fp32.  A
// quotient by 127 of a value with 8 significant bits is either exact or has an
// endless periodic binary expansion, so it never lies exactly between two
// fp32 values: the correctly rounded division equals rounding the exact value.
__device__ __forceinline__ float i8_row_scale(float amax) { return __fdiv_rn(amax, 127.f); }

// The code of x for a row scale > 0 (inv = 1 / scale, rounded).  The rounded
// quotient proposes floor(|x| / scale); the sign of |x| - (n + 1/2) scale,
// taken exactly by one fused multiply-add, decides between n and n + 1 (the
// proposal can be one off only next to an integer, far from that midpoint).
// Scales below 2^-100 are lifted by 2^64 first (exact), which keeps the
// difference out of the fp32 subnormals where a nonzero value could round to 0.
__device__ __forceinline__ int i8_quantize(float x, float scale, float inv) {
    float a = fabsf(x), s = scale;
    float q;
    if (s < 0x1p-100f) {
        a *= 0x1p64f;
        s *= 0x1p64f;
        q = __fdiv_rn(a, s);
    } else {
        q = __fmul_rn(a, inv);
    }
    const float n = fminf(floorf(q), 127.f);
    const float d = __fmaf_rn(-(n + 0.5f), s, a);  // sign of a - (n + 1/2) s, exactly
    int r = int(n);
    if (d > 0.f || (d == 0.f && (r & 1))) ++r;
    r = min(r, 127);
    return x < 0.f ? -r : r;
}

// Four codes (the bytes of w, lowest first) as two bf16x2 pairs: every integer
// in [-127, 127] is exact in bf16.
__device__ __forceinline__ uint2 i8x4_bf16x4(uint32_t w) {
    const float c0 = float(int(w << 24) >> 24), c1 = float(int(w << 16) >> 24);
    const float c2 = float(int(w << 8) >> 24), c3 = float(int(w) >> 24);
    return make_uint2(pack_bf2(c0, c1), pack_bf2(c2, c3));
}

}  // namespace lcsw
