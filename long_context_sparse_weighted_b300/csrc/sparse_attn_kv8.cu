// Sparse attention over an FP8 (E4M3) K/V cache: one fp32 scale per token
// row, the element value e4m3(code) * scale (the serving stack of the reading
// notes "GLM-5.3-Flash: Hybrid Attention, IndexPool, and Vision-in-the-Loop"
// quantizes caches per tier to INT8, FP8 or BF16, section "The serving
// stack"; the format is the one of the FP8 pooled keys, e4m3_core.cuh).
//
//   z_j = scale * ks_j * (q . e4m3(kc_j)),   out = sum_j softmax_j(z) vs_j e4m3(vc_j)
//
// The split-K structure of sparse_attn.cu, with the gather halved: a chunk's
// codes (DQK + DV bytes a token, against 2 (DQK + DV) in bf16) and its two
// scales land in a staging buffer by 16-byte cp.async, and the block widens
// the codes to bf16 tiles (exactly: an E4M3 value has four significant bits)
// while the next chunk's codes are in flight.  The scores of a token are then
// multiplied by its key scale, and its softmax weight by its value scale in
// the P V product (attn_core.cuh), so neither scale is rounded into the tiles.
//
// The INT8 tier (I8 = true, i8_core.cuh) runs the same kernel: its codes are
// integers in [-127, 127], which bf16 also holds exactly, with one fp32 scale
// per token row (amax / 127).
#include "attn_core.cuh"
#include "common.cuh"
#include "e4m3_core.cuh"
#include "i8_core.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

constexpr int kThr8 = 128;
constexpr int kHeadGroup8 = 64;
constexpr int kTarget8 = 296;
constexpr float kLog2e8 = 1.4426950408889634f;
constexpr float kLn28 = 0.6931471805599453f;

template <int DQK, int DV>
struct Kv8Smem {
    static constexpr int QP = DQK + 8, VP = DV + 8;
    static constexpr int q_bytes = kHeadGroup8 * QP * 2;
    static constexpr int k_bytes = kChunk * QP * 2;
    static constexpr int v_bytes = kChunk * VP * 2;
    static constexpr int tiles = k_bytes + v_bytes;                // one bf16 chunk
    static constexpr int stage = kChunk * (DQK + DV) + 2 * kChunk * 4;  // codes + scales
    static constexpr int state_bytes = 4 * 16 * (DV + 2) * 4;
    static constexpr int body = tiles + 2 * stage > state_bytes ? tiles + 2 * stage : state_bytes;
    static constexpr int total = q_bytes + body + 2 * kChunk * 4;
};

// One chunk's codes and scales into staging buffer `sb`: groups glist[0..n)
// of a sequence with complete groups [0, G); missing or invalid groups are
// zero-filled (codes and scales) and get id -1.
template <int DQK, int DV>
__device__ __forceinline__ void gather_codes(unsigned char *sb, int *sg, const int32_t *glist,
                                             int n, int P, int G, const uint8_t *kcb,
                                             const float *ksb, const uint8_t *vcb,
                                             const float *vsb) {
    const int tid = threadIdx.x;
    uint8_t *kc = sb;
    uint8_t *vc = sb + kChunk * DQK;
    float *ks = reinterpret_cast<float *>(sb + kChunk * (DQK + DV));
    float *vs = ks + kChunk;
    const int gpc = kChunk / P;
    if (tid < gpc) {
        const int g = tid < n ? glist[tid] : -1;
        sg[tid] = (g >= 0 && g < G) ? g : -1;
    }
    auto token = [&](int tr, int64_t &row) {
        const int q = tr / P;
        const int g = q < n ? glist[q] : -1;
        row = int64_t(g) * P + tr % P;
        return g >= 0 && g < G;
    };
    for (int e = tid; e < kChunk * (DQK / 16); e += kThr8) {
        const int tr = e / (DQK / 16), c16 = e % (DQK / 16);
        int64_t row;
        const bool ok = token(tr, row);
        cp_async16(smem_u32(kc + tr * DQK + c16 * 16), ok ? kcb + row * DQK + c16 * 16 : kcb,
                   ok ? 16 : 0);
    }
    for (int e = tid; e < kChunk * (DV / 16); e += kThr8) {
        const int tr = e / (DV / 16), c16 = e % (DV / 16);
        int64_t row;
        const bool ok = token(tr, row);
        cp_async16(smem_u32(vc + tr * DV + c16 * 16), ok ? vcb + row * DV + c16 * 16 : vcb,
                   ok ? 16 : 0);
    }
    for (int tr = tid; tr < 2 * kChunk; tr += kThr8) {
        const int t = tr % kChunk;
        int64_t row;
        const bool ok = token(t, row);
        const float *src = tr < kChunk ? ksb : vsb;
        float *dst = tr < kChunk ? ks + t : vs + t;
        if (ok) {
            cp_async4(smem_u32(dst), src + row);
        } else {
            *dst = 0.f;  // a masked token's weight is 0 and must stay finite
        }
    }
    cp_async_commit();
}

// Four codes (one word) -> four bf16 values, exactly.
template <bool I8>
__device__ __forceinline__ uint2 widen4(uint32_t w) {
    if constexpr (I8) return i8x4_bf16x4(w);
    else return make_uint2(e4m3x2_bf16x2(w), e4m3x2_bf16x2(w >> 16));
}

// Codes of staging buffer `sb` -> bf16 K and V tiles (row pitches QP, VP).
template <int DQK, int DV, bool I8>
__device__ __forceinline__ void widen_codes(const unsigned char *sb, uint16_t *sk, uint16_t *sv,
                                            int QP, int VP) {
    const uint8_t *kc = sb;
    const uint8_t *vc = sb + kChunk * DQK;
    for (int e = threadIdx.x; e < kChunk * (DQK / 4); e += kThr8) {
        const int tr = e / (DQK / 4), c4 = e % (DQK / 4);
        const uint32_t w = *reinterpret_cast<const uint32_t *>(kc + tr * DQK + c4 * 4);
        *reinterpret_cast<uint2 *>(sk + tr * QP + c4 * 4) = widen4<I8>(w);
    }
    for (int e = threadIdx.x; e < kChunk * (DV / 4); e += kThr8) {
        const int tr = e / (DV / 4), c4 = e % (DV / 4);
        const uint32_t w = *reinterpret_cast<const uint32_t *>(vc + tr * DV + c4 * 4);
        *reinterpret_cast<uint2 *>(sv + tr * VP + c4 * 4) = widen4<I8>(w);
    }
}

template <int DQK, int DV, bool I8>
__global__ void __launch_bounds__(kThr8) sparse_attn_kv8_kernel(
    const uint16_t *__restrict__ q, const uint8_t *__restrict__ kc, int64_t skc_b,
    const float *__restrict__ ks, int64_t sks_b, const uint8_t *__restrict__ vc, int64_t svc_b,
    const float *__restrict__ vs, int64_t svs_b, const int32_t *__restrict__ seq_len,
    const int32_t *__restrict__ idx, int T, int H_q, int P, int k, int S, float scale_log2,
    uint16_t *__restrict__ out, float *__restrict__ lse, float *__restrict__ part_o,
    float2 *__restrict__ part_ml) {
    using L = Kv8Smem<DQK, DV>;
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *sq = reinterpret_cast<uint16_t *>(smem);
    uint16_t *sk = reinterpret_cast<uint16_t *>(smem + L::q_bytes);
    uint16_t *sv = reinterpret_cast<uint16_t *>(smem + L::q_bytes + L::k_bytes);
    unsigned char *stage = smem + L::q_bytes + L::tiles;          // [2][L::stage]
    float *state = reinterpret_cast<float *>(smem + L::q_bytes);
    int *sgrp = reinterpret_cast<int *>(smem + L::q_bytes + L::body);  // [2][kChunk]

    const int s = blockIdx.x;
    const int64_t row = blockIdx.y;
    const int hg0 = blockIdx.z * kHeadGroup8;
    const int HG = min(kHeadGroup8, H_q - hg0);
    const int b = int(row / T);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int G = __ldg(seq_len + b) / P;
    const int gps = (k + S - 1) / S;
    const int j0 = s * gps, j1 = min(k, j0 + gps);
    const int gpc = kChunk / P;
    const int nchunks = j1 > j0 ? (j1 - j0 + gpc - 1) / gpc : 0;
    const int32_t *irow = idx + row * k;
    const uint8_t *kcb = kc + int64_t(b) * skc_b;
    const uint8_t *vcb = vc + int64_t(b) * svc_b;
    const float *ksb = ks + int64_t(b) * sks_b;
    const float *vsb = vs + int64_t(b) * svs_b;

    const int MT = HG / 16, TS = 4 / MT;
    const int mt = warp % MT, ts = warp / MT;
    const int ntok = kChunk / TS, tok0 = ts * ntok;

    const uint16_t *qrow = q + (row * H_q + hg0) * DQK;
    for (int p = tid; p < HG * (DQK / 8); p += kThr8) {
        const int h = p / (DQK / 8), c8 = p % (DQK / 8);
        *reinterpret_cast<uint4 *>(sq + h * L::QP + c8 * 8) = ld_nc16(qrow + int64_t(h) * DQK + c8 * 8);
    }
    auto issue = [&](int ci) {
        const int jb = j0 + ci * gpc;
        gather_codes<DQK, DV>(stage + (ci & 1) * L::stage, sgrp + (ci & 1) * kChunk, irow + jb,
                              min(gpc, j1 - jb), P, G, kcb, ksb, vcb, vsb);
    };
    if (nchunks > 0) issue(0);
    __syncthreads();  // Q in shared

    uint32_t qa[DQK / 16][4];
    load_q_frags<DQK>(qa, sq, L::QP, mt);
    AttnWarpState<DV> st;
    st.init();
    for (int ci = 0; ci < nchunks; ++ci) {
        if (ci + 1 < nchunks) {
            issue(ci + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // chunk ci's codes landed; every warp is done with the tiles
        const unsigned char *sb = stage + (ci & 1) * L::stage;
        widen_codes<DQK, DV, I8>(sb, sk, sv, L::QP, L::VP);
        __syncthreads();
        const float *kscale = reinterpret_cast<const float *>(sb + kChunk * (DQK + DV));
        attn_chunk<DQK, DV>(st, qa, sk, sv, sgrp + (ci & 1) * kChunk, L::QP, L::VP, P, tok0,
                            ntok, scale_log2, nullptr, 0, kscale, kscale + kChunk);
        __syncthreads();  // the tiles and this staging buffer are reused
    }
    store_warp_state<DV>(st, state + warp * 16 * (DV + 2));
    __syncthreads();
    for (int p = tid; p < HG * (DV / 2); p += kThr8) {
        const int hl = p / (DV / 2), d2 = (p % (DV / 2)) * 2;
        float Lsum;
        const float4 r = merge_states<DV>(state, MT, TS, hl, d2, Lsum);
        const int h = hg0 + hl;
        if (S == 1) {
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            *reinterpret_cast<uint32_t *>(out + (row * H_q + h) * DV + d2) =
                pack_bf2(r.z * inv, r.w * inv);
            if (lse && d2 == 0)
                lse[row * H_q + h] = Lsum > 0.f ? (r.x + log2f(Lsum)) * kLn28 : -INFINITY;
        } else {
            const int64_t pi = (row * S + s) * H_q + h;
            *reinterpret_cast<float2 *>(part_o + pi * DV + d2) = make_float2(r.z, r.w);
            if (d2 == 0) part_ml[pi] = make_float2(r.x, Lsum);
        }
    }
}

template <int DQK, int DV, bool I8>
cudaError_t launch_kv8_typed(const uint16_t *q, const uint8_t *kc, int64_t skc_b, const float *ks,
                             int64_t sks_b, const uint8_t *vc, int64_t svc_b, const float *vs,
                             int64_t svs_b, const int32_t *seq_len, const int32_t *idx, int B,
                             int T, int H_q, int P, int k, float scale, uint16_t *out, float *lse,
                             void *ws, cudaStream_t st) {
    const int64_t rows = int64_t(B) * T;
    const int S = sparse_attn_kv8_splits(rows, H_q, k, P);
    const int HGs = (H_q + kHeadGroup8 - 1) / kHeadGroup8;
    using L = Kv8Smem<DQK, DV>;
    auto kern = sparse_attn_kv8_kernel<DQK, DV, I8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
    if (e != cudaSuccess) return e;
    float *part_o = reinterpret_cast<float *>(ws);
    float2 *part_ml = reinterpret_cast<float2 *>(
        reinterpret_cast<char *>(ws) + size_t(rows) * S * H_q * DV * sizeof(float));
    if (rows > 65535) return cudaErrorInvalidConfiguration;
    kern<<<dim3(S, unsigned(rows), HGs), kThr8, L::total, st>>>(
        q, kc, skc_b, ks, sks_b, vc, svc_b, vs, svs_b, seq_len, idx, T, H_q, P, k, S,
        scale * kLog2e8, out, lse, part_o, part_ml);
    e = cudaGetLastError();
    if (e != cudaSuccess || S == 1) return e;
    splitk_combine_kernel<DV><<<dim3(unsigned(rows), (H_q + 7) / 8), 256, 0, st>>>(
        part_o, part_ml, H_q, S, out, lse);
    return cudaGetLastError();
}

}  // namespace

int sparse_attn_kv8_splits(int64_t rows, int H_q, int k, int P) {
    const int64_t HGs = (H_q + kHeadGroup8 - 1) / kHeadGroup8;
    const int64_t chunks = (int64_t(k) * P + kChunk - 1) / kChunk;
    int64_t want = (kTarget8 + rows * HGs - 1) / (rows * HGs);
    if (want > chunks) want = chunks;
    if (want < 1) want = 1;
    return int(want);
}

size_t sparse_attn_kv8_ws_bytes(int64_t rows, int H_q, int d_v, int k, int P) {
    const int S = sparse_attn_kv8_splits(rows, H_q, k, P);
    if (S == 1) return 0;
    return size_t(rows) * S * H_q * (size_t(d_v) * sizeof(float) + sizeof(float2));
}

cudaError_t launch_sparse_attn_kv8(const uint16_t *q, const uint8_t *kc, int64_t skc_b,
                                   const float *ks, int64_t sks_b, const uint8_t *vc,
                                   int64_t svc_b, const float *vs, int64_t svs_b,
                                   const int32_t *seq_len, const int32_t *idx, int B, int T,
                                   int H_q, int d_qk, int d_v, int P, int k, float scale,
                                   uint16_t *out, float *lse, void *ws, bool int8_codes,
                                   cudaStream_t st) {
    if (int64_t(B) * T == 0) return cudaSuccess;
#define LCSW_KV8(DQ, DVV)                                                                     \
    if (d_qk == DQ && d_v == DVV)                                                            \
        return int8_codes                                                                     \
                   ? launch_kv8_typed<DQ, DVV, true>(q, kc, skc_b, ks, sks_b, vc, svc_b, vs,   \
                                                     svs_b, seq_len, idx, B, T, H_q, P, k,    \
                                                     scale, out, lse, ws, st)                 \
                   : launch_kv8_typed<DQ, DVV, false>(q, kc, skc_b, ks, sks_b, vc, svc_b, vs,  \
                                                      svs_b, seq_len, idx, B, T, H_q, P, k,   \
                                                      scale, out, lse, ws, st);
    LCSW_KV8(64, 64)
    LCSW_KV8(128, 64)
    LCSW_KV8(128, 128)
    LCSW_KV8(192, 128)
    LCSW_KV8(192, 64)
    LCSW_KV8(64, 128)
#undef LCSW_KV8
    return cudaErrorInvalidValue;
}

}  // namespace lcsw
