// Exact IndexPool arithmetic (shared by the pooling kernel and the fused
// decode step, so both produce the same bits): sum_j alpha_j * k_j formed with
// error-free fp32 transformations and rounded once to bf16 (nearest even).
#pragma once

#include "common.cuh"

namespace lcsw {

// a*b == p + e exactly (fp32 has a fused multiply-add).
__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e) {
    p = __fmul_rn(a, b);
    e = __fmaf_rn(a, b, -p);
}

// a+b == s + e exactly (Knuth's branch-free two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Nearest bf16 (ties to even) of hi + lo, where hi = fl(hi + lo).  The bf16
// grid is a subset of the fp32 grid, so rounding hi gives the right answer
// unless hi sits exactly on a bf16 midpoint while lo != 0; then lo says on
// which side of the midpoint the exact value lies.
__device__ __forceinline__ uint32_t round_bf16_exact(float hi, float lo) {
    uint32_t u = __float_as_uint(hi);
    if ((u & 0xFFFFu) == 0x8000u && lo != 0.0f) {
        bool away = (lo > 0.0f) == (hi > 0.0f);
        return (u >> 16) + (away ? 1u : 0u);
    }
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

template <int P>
__device__ __forceinline__ uint32_t pool_pair(const float (&a)[P], const uint32_t (&w)[P],
                                              bool high) {
    float s = 0.0f, c = 0.0f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
        float kv = high ? bf_hi(w[j]) : bf_lo(w[j]);
        float p, e, t, err;
        two_prod(a[j], kv, p, e);
        two_sum(s, p, t, err);
        s = t;
        c = __fadd_rn(c, __fadd_rn(err, e));
    }
    float hi, lo;
    two_sum(s, c, hi, lo);
    return round_bf16_exact(hi, lo);
}

// Pool 8 dims (one 16-byte chunk of each of the P source rows).
template <int P>
__device__ __forceinline__ uint4 pool_chunk(const float (&a)[P], const uint4 (&rows)[P]) {
    uint32_t wx[P], wy[P], wz[P], ww[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        wx[j] = rows[j].x;
        wy[j] = rows[j].y;
        wz[j] = rows[j].z;
        ww[j] = rows[j].w;
    }
    uint4 o;
    o.x = pool_pair<P>(a, wx, false) | (pool_pair<P>(a, wx, true) << 16);
    o.y = pool_pair<P>(a, wy, false) | (pool_pair<P>(a, wy, true) << 16);
    o.z = pool_pair<P>(a, wz, false) | (pool_pair<P>(a, wz, true) << 16);
    o.w = pool_pair<P>(a, ww, false) | (pool_pair<P>(a, ww, true) << 16);
    return o;
}

// One pooled key from its P rows and weights staged in shared memory
// (rows_s: [P][64] bf16, w_s: [P]): lanes 0-7 each pool 8 dims and store them
// to `dst_s` (shared) and, unless null, `dst` (global).  Out of line: it runs
// once per call.
static __device__ __noinline__ void pool_staged(int P, const uint16_t *rows_s, const float *w_s, int lane,
                                         uint16_t *dst_s, uint16_t *dst) {
    if (lane >= 8) return;
    uint4 o;
#define LCSW_POOL_STAGED(PP)                                                              \
    {                                                                                     \
        uint4 rows[PP];                                                                   \
        float a[PP];                                                                      \
        for (int j = 0; j < PP; ++j) {                                                    \
            rows[j] = *reinterpret_cast<const uint4 *>(rows_s + j * 64 + lane * 8);       \
            a[j] = w_s[j];                                                                \
        }                                                                                 \
        o = pool_chunk<PP>(a, rows);                                                      \
    }
    if (P == 1) LCSW_POOL_STAGED(1)
    else if (P == 2) LCSW_POOL_STAGED(2)
    else if (P == 4) LCSW_POOL_STAGED(4)
    else LCSW_POOL_STAGED(8)
#undef LCSW_POOL_STAGED
    *reinterpret_cast<uint4 *>(dst_s + lane * 8) = o;
    if (dst) *reinterpret_cast<uint4 *>(dst + lane * 8) = o;
}

}  // namespace lcsw
