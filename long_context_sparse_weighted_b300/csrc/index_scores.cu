// Lightweight multi-head indexer, decode form (reading notes "GLM-5.3-Flash:
// Hybrid Attention, IndexPool, and Vision-in-the-Loop", section 2: a
// lightweight indexer pulls the relevant slices out of the window; DSA
// indexer form):
//
//   s[b][t][g] = sum_h w[b][t][h] * max(0, q[b][t][h][:] . kbar[b][g][:])
//
// Decode reads every pooled key once (128 bytes) and does 8 x 64 MACs with
// it, which at HBM rate is more than the fp32 CUDA cores can issue, so the
// dot products run on the tensor cores (mma.sync m16n8k16, bf16 x bf16 ->
// fp32): A = 16 pooled keys x 16 dims, B = 16 dims x 8 heads.
//
// The key rows go from HBM straight into A-fragment registers with no
// shared-memory staging.  Because the contraction index can be permuted
// freely (the same way for A and B), lane (r = lane/4, c = lane%4) loads the
// 16-byte chunks c and 4+c of rows r and r+8 of a 16-key tile: each load
// instruction of the warp covers 8 rows x 64 contiguous bytes, so every
// 32-byte sector it touches is used in full.  Word i of the chunk feeds
// k-step (2*half + i/2); the query fragments use the same map.
#include "common.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

constexpr int kDIdx = 64;

template <int NT, int TQ>
__global__ void __launch_bounds__(256) index_scores_mma_kernel(
    const uint16_t *__restrict__ q_idx, const float *__restrict__ w_head,
    const uint16_t *__restrict__ k_pooled, int64_t sp_b, const int32_t *__restrict__ seq_len,
    const int32_t *__restrict__ q_pos, int T, int H_i, int P, int G_max,
    float *__restrict__ scores) {
    const int qb_per_b = (T + TQ - 1) / TQ;
    const int b = blockIdx.y / qb_per_b;
    const int t0 = (blockIdx.y % qb_per_b) * TQ;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, c = lane & 3;
    const int G = __ldg(seq_len + b) / P;

    int nvis[TQ];
    uint32_t bq[TQ][NT][4][2];
    float wv[TQ][NT][2];
    int nvis_max = 0;
#pragma unroll
    for (int t = 0; t < TQ; ++t) {
        const int tt = t0 + t;
        const bool tv = tt < T;
        int nv = 0;
        if (tv) {
            nv = G;
            if (q_pos) {
                const int p = __ldg(q_pos + int64_t(b) * T + tt);
                const int m = p < 0 ? 0 : (p + 1) / P;
                nv = m < nv ? m : nv;
            }
        }
        nv = nv < G_max ? nv : G_max;  // never read past the cache's allocated rows
        nvis[t] = nv;
        nvis_max = nv > nvis_max ? nv : nvis_max;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int head = nt * 8 + r;
            uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
            if (tv && head < H_i) {
                const uint16_t *qp = q_idx + ((int64_t(b) * T + tt) * H_i + head) * kDIdx;
                h0 = ld_nc16(qp + 8 * c);
                h1 = ld_nc16(qp + 32 + 8 * c);
            }
            bq[t][nt][0][0] = h0.x; bq[t][nt][0][1] = h0.y;
            bq[t][nt][1][0] = h0.z; bq[t][nt][1][1] = h0.w;
            bq[t][nt][2][0] = h1.x; bq[t][nt][2][1] = h1.y;
            bq[t][nt][3][0] = h1.z; bq[t][nt][3][1] = h1.w;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = nt * 8 + 2 * c + e;
                wv[t][nt][e] = (tv && h < H_i) ? __ldg(w_head + (int64_t(b) * T + tt) * H_i + h)
                                               : 0.0f;
            }
        }
    }

    const int wpb = blockDim.x >> 5;
    const int tiles = (G_max + 15) >> 4;
    const uint16_t *kb = k_pooled + int64_t(b) * sp_b;
    for (int tile = blockIdx.x * wpb + warp; tile < tiles; tile += gridDim.x * wpb) {
        const int ga = tile * 16 + r, gb = ga + 8;
        const uint4 z = make_uint4(0, 0, 0, 0);
        uint4 a_lo = z, a_hi = z, b_lo = z, b_hi = z;
        if (ga < nvis_max) {
            a_lo = ld_stream16(kb + int64_t(ga) * kDIdx + 8 * c);
            a_hi = ld_stream16(kb + int64_t(ga) * kDIdx + 32 + 8 * c);
        }
        if (gb < nvis_max) {
            b_lo = ld_stream16(kb + int64_t(gb) * kDIdx + 8 * c);
            b_hi = ld_stream16(kb + int64_t(gb) * kDIdx + 32 + 8 * c);
        }
        const uint32_t A0[4] = {a_lo.x, a_lo.z, a_hi.x, a_hi.z};  // row r,   k-lo of step s
        const uint32_t A2[4] = {a_lo.y, a_lo.w, a_hi.y, a_hi.w};  // row r,   k-hi
        const uint32_t A1[4] = {b_lo.x, b_lo.z, b_hi.x, b_hi.z};  // row r+8, k-lo
        const uint32_t A3[4] = {b_lo.y, b_lo.w, b_hi.y, b_hi.w};  // row r+8, k-hi
#pragma unroll
        for (int t = 0; t < TQ; ++t) {
            if (t0 + t >= T) break;
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_bf16_16816(acc[nt], A0[s], A1[s], A2[s], A3[s], bq[t][nt][s][0],
                                   bq[t][nt][s][1]);
            float pa = 0.f, pb = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                pa = __fadd_rn(pa, __fmul_rn(wv[t][nt][0], fmaxf(acc[nt][0], 0.f)));
                pa = __fadd_rn(pa, __fmul_rn(wv[t][nt][1], fmaxf(acc[nt][1], 0.f)));
                pb = __fadd_rn(pb, __fmul_rn(wv[t][nt][0], fmaxf(acc[nt][2], 0.f)));
                pb = __fadd_rn(pb, __fmul_rn(wv[t][nt][1], fmaxf(acc[nt][3], 0.f)));
            }
            pa = __fadd_rn(pa, __shfl_xor_sync(0xffffffffu, pa, 1));
            pb = __fadd_rn(pb, __shfl_xor_sync(0xffffffffu, pb, 1));
            pa = __fadd_rn(pa, __shfl_xor_sync(0xffffffffu, pa, 2));
            pb = __fadd_rn(pb, __shfl_xor_sync(0xffffffffu, pb, 2));
            float *srow = scores + (int64_t(b) * T + t0 + t) * G_max;
            if (c == 0 && ga < G_max) srow[ga] = ga < nvis[t] ? __fadd_rn(pa, 0.0f) : -INFINITY;
            if (c == 1 && gb < G_max) srow[gb] = gb < nvis[t] ? __fadd_rn(pb, 0.0f) : -INFINITY;
        }
    }
}

__global__ void visible_counts_kernel(const int32_t *__restrict__ seq_len,
                                      const int32_t *__restrict__ q_pos, int B, int T, int P,
                                      int32_t *__restrict__ n_valid) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= int64_t(B) * T) return;
    const int b = int(i / T);
    int n = seq_len[b] / P;
    if (q_pos) {
        const int p = q_pos[i];
        const int m = p < 0 ? 0 : (p + 1) / P;
        n = m < n ? m : n;
    }
    n_valid[i] = n;
}

__global__ void prefill_positions_kernel(const int32_t *__restrict__ seq_len, int B, int T,
                                         int32_t *__restrict__ q_pos) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= int64_t(B) * T) return;
    const int b = int(i / T), t = int(i % T);
    q_pos[i] = seq_len[b] - T + t;
}

}  // namespace

cudaError_t launch_prefill_positions(const int32_t *seq_len, int B, int T, int32_t *q_pos,
                                     cudaStream_t st) {
    const int64_t n = int64_t(B) * T;
    if (n == 0) return cudaSuccess;
    prefill_positions_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(seq_len, B, T, q_pos);
    return cudaGetLastError();
}

cudaError_t launch_index_scores_mma(const uint16_t *q_idx, const float *w_head,
                                    const uint16_t *k_pooled, int64_t sp_b,
                                    const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                    int H_i, int P, int G_max, float *scores, cudaStream_t st) {
    if (B == 0 || T == 0 || G_max == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int TQ = (T == 1) ? 1 : 4;
    const int64_t gy = int64_t(B) * ((T + TQ - 1) / TQ);
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    const int threads = 256, wpb = threads / 32;
    const int64_t tiles = (G_max + 15) / 16;
    int64_t gx = (tiles + wpb - 1) / wpb;
    int64_t want = (int64_t(sms) * 8 + gy - 1) / gy;
    if (want < 1) want = 1;
    if (gx > want) gx = want;
    dim3 grid((unsigned)gx, (unsigned)gy);
    const int NT = H_i > 8 ? 2 : 1;
#define LCSW_IS(NTT, TQQ)                                                              \
    index_scores_mma_kernel<NTT, TQQ><<<grid, threads, 0, st>>>(                      \
        q_idx, w_head, k_pooled, sp_b, seq_len, q_pos, T, H_i, P, G_max, scores)
    if (NT == 1 && TQ == 1) LCSW_IS(1, 1);
    else if (NT == 1) LCSW_IS(1, 4);
    else if (TQ == 1) LCSW_IS(2, 1);
    else LCSW_IS(2, 4);
#undef LCSW_IS
    return cudaGetLastError();
}

cudaError_t launch_visible_counts(const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                  int P, int32_t *n_valid, cudaStream_t st) {
    const int64_t n = int64_t(B) * T;
    if (n == 0) return cudaSuccess;
    visible_counts_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(seq_len, q_pos, B, T, P,
                                                                      n_valid);
    return cudaGetLastError();
}

}  // namespace lcsw
