// FP8 (OCP E4M3) pooled indexer keys and queries: one fp32 scale per 64-value
// row, codes rounded to nearest with ties to the even code, saturating at
// +-448.  The serving stack of the reading notes ("GLM-5.3-Flash: Hybrid
// Attention, IndexPool, and Vision-in-the-Loop", section "The serving stack")
// quantizes caches per tier to INT8, FP8 or BF16 and says nothing more about
// the format; this is the plainest reading:
//
//   scale = amax(|x|) / 448 (fp32),  code_i = e4m3(x_i / scale)  (0 if scale = 0)
//
// The rounding decision is exact: an fp32 quotient proposes a code, and the
// sign of x - m * scale, with m the midpoint between that code and its
// neighbour on the quotient's side, settles it (an FMA forms that difference
// with one rounding, which keeps its sign).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace lcsw {

// The FP8 pooled-key cache, per sequence: tiles of 16 groups, each 16 rows of
// 64 codes followed by the 16 rows' fp32 scales.
constexpr int kE4m3TileBytes = 16 * 64 + 16 * 4;

// Value of a code (sign, 4 exponent bits with bias 7, 3 mantissa bits; the
// exponent field 0 holds the subnormals m * 2^-9).  Codes 0x7F/0xFF (NaN) are
// never produced.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
    const float mag = e == 0u ? float(m) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (c & 0x80u) ? -mag : mag;
}

// Nearest code of x / scale (scale > 0; inv = 1 / scale, rounded), ties to
// the even code, saturating.  The quotient only proposes a code: within a
// few ulps of the exact one, it lands on the right code or its neighbour,
// and the midpoint test below decides between them.
__device__ __forceinline__ uint32_t e4m3_quantize(float x, float scale, float inv) {
    const uint32_t sign = (__float_as_uint(x) >> 24) & 0x80u;
    const float a = fabsf(x);
    // (a scale too small for its reciprocal to be finite takes the division)
    const float q = isinf(inv) ? __fdiv_rn(a, scale) : __fmul_rn(a, inv);
    if (q >= 448.f) return sign | 0x7Eu;
    // proposed code from the rounded quotient
    uint32_t c;
    {
        unsigned short pair;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.f), "f"(q));
        c = pair & 0x7Fu;
    }
    const float v = e4m3_value(c);
    if (q == v) return sign | c;  // the exact quotient is within a few ulps of the code v
    // midpoint between c and its neighbour on the quotient's side
    const uint32_t lo = q > v ? c : c - 1u, hi = lo + 1u;
    const float mid = 0.5f * (e4m3_value(lo) + e4m3_value(hi));
    const float d = __fmaf_rn(-mid, scale, a);  // sign of a - mid * scale, exactly
    uint32_t r;
    if (d > 0.f) r = hi;
    else if (d < 0.f) r = lo;
    else r = (lo & 1u) ? hi : lo;
    return sign | min(r, 0x7Eu);
}

// Two E4M3 codes (bits 0-15 of w, the lower code in bits 0-7) as an f16x2 pair;
// every E4M3 value is exact in f16.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t w) {
    uint32_t r;
    asm("{\n .reg .b16 t;\n mov.b16 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
        : "=r"(r)
        : "h"((unsigned short)(w & 0xFFFFu)));
    return r;
}

// The same two codes as a bf16x2 pair (also exact: an E4M3 value has at most
// four significant bits and lies inside the bf16 range).
__device__ __forceinline__ uint32_t e4m3x2_bf16x2(uint32_t w) {
    const uint32_t h = e4m3x2_f16x2(w);
    const float lo = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
    const float hi = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
    return pack_bf2(lo, hi);
}

// Scale of a row from its largest magnitude: amax / 448 rounded to fp32 (the
// same value as rounding the double quotient: amax has 8 significant bits, and
// a quotient by 7 * 2^6 never lands exactly between two fp32 values).
__device__ __forceinline__ float e4m3_row_scale(float amax) { return __fdiv_rn(amax, 448.f); }

}  // namespace lcsw
