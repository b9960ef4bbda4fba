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

// The same correctly rounded value by a shorter route when it is safe: an fp32
// fma chain s approximates the exact sum X with |s - X| <= E, where E comes
// from the chain of magnitudes m = sum |alpha_j k_j| (each fma rounds once,
// relative 2^-24, so |s - X| <= P 2^-24 m (1 + 2^-24)^(2P) plus underflow,
// below (P + 1) 2^-24 m + 2^-140).  If no bf16 rounding boundary lies within
// E of s -- the midpoint between the two bf16 values around s, and a quarter
// bf16 step for the boundaries beyond them -- X rounds like s.  Returns false
// (undecided) otherwise, and for zero, subnormal or non-finite s.
template <int P>
__device__ __forceinline__ bool pool_pair_fast(const float (&a)[P], const uint32_t (&w)[P],
                                               bool high, uint32_t &out) {
    float s = 0.0f, m = 0.0f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
        const float kv = high ? bf_hi(w[j]) : bf_lo(w[j]);
        s = __fmaf_rn(a[j], kv, s);
        m = __fmaf_rn(fabsf(a[j]), fabsf(kv), m);
    }
    const float E = __fmaf_rn(m, float(P + 1) * 0x1p-24f, 0x1p-140f);
    const uint32_t u = __float_as_uint(s);
    const float lo = __uint_as_float(u & 0xFFFF0000u);          // s truncated to bf16
    const float mid = __uint_as_float((u & 0xFFFF0000u) | 0x8000u);
    // s - mid is exact (same sign and exponent); |lo| / 1024 is at most a
    // quarter of the bf16 step at s
    const float room = fminf(fabsf(__fsub_rn(s, mid)), fabsf(lo) * 0x1p-10f);
    out = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    return E < room;
}

template <int P>
__device__ __forceinline__ uint32_t pool_pair_any(const float (&a)[P], const uint32_t (&w)[P],
                                                  bool high) {
    uint32_t r;
    if (pool_pair_fast<P>(a, w, high, r)) return r;
    return pool_pair<P>(a, w, high);
}

// Pool 8 dims (one 16-byte chunk of each of the P source rows) through the
// shorter route where it decides the rounding.
template <int P>
__device__ __forceinline__ uint4 pool_chunk_fast(const float (&a)[P], const uint4 (&rows)[P]) {
    uint32_t wx[P], wy[P], wz[P], ww[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        wx[j] = rows[j].x;
        wy[j] = rows[j].y;
        wz[j] = rows[j].z;
        ww[j] = rows[j].w;
    }
    uint4 o;
    o.x = pool_pair_any<P>(a, wx, false) | (pool_pair_any<P>(a, wx, true) << 16);
    o.y = pool_pair_any<P>(a, wy, false) | (pool_pair_any<P>(a, wy, true) << 16);
    o.z = pool_pair_any<P>(a, wz, false) | (pool_pair_any<P>(a, wz, true) << 16);
    o.w = pool_pair_any<P>(a, ww, false) | (pool_pair_any<P>(a, ww, true) << 16);
    return o;
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
